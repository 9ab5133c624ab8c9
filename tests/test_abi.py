"""The C-ABI library: it builds, loads without a GPU, exports every declared
symbol, and rejects bad arguments on the host before touching CUDA."""

import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "moe_a16w4.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[a-z_0-9 ]*?\**\s*(\w+)\s*\(", text, flags=re.M)
    return sorted({n for n in names if n.startswith(("moe_", "requant_"))})


@pytest.fixture(scope="module")
def lib():
    from mxfp4_weight_only_gb300 import _native, build

    build.build()
    return _native.load()


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("moe_a16w4_mxfp4", "moe_a16w4_int4g32", "requant_mxfp4_to_int4g32", "moe_workspace_bytes",
              "moe_route", "moe_read_status", "moe_error_string", "moe_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from mxfp4_weight_only_gb300 import _native

    for n in _declared_functions():
        assert hasattr(lib, n), n
        assert n in _native.SIGNATURES, n


def test_checked_library_exports_every_declared_symbol(lib):
    from mxfp4_weight_only_gb300 import _native, build

    checked = _native.load(checked=True)
    assert checked is not lib and checked._name == build.lib_path(checked=True)
    for n in _declared_functions():
        assert hasattr(checked, n), n
    assert checked.moe_abi_version() == lib.moe_abi_version()


def test_version_and_error_strings(lib):
    assert lib.moe_abi_version() == 104
    assert lib.moe_error_string(0) == b"ok"
    assert b"SwiGLU" in lib.moe_error_string(-4)


def test_workspace_bytes_host_logic(lib):
    from mxfp4_weight_only_gb300 import dims

    d1 = dims(112, 3584, 3072, 15, 1)
    d32 = dims(112, 3584, 3072, 15, 32)
    assert 0 < lib.moe_workspace_bytes(ctypes.byref(d1)) < lib.moe_workspace_bytes(ctypes.byref(d32))
    assert lib.moe_workspace_bytes(ctypes.byref(dims(112, 3584 + 32, 3072, 15, 1))) == 0  # H % 64
    assert lib.moe_workspace_bytes(ctypes.byref(dims(0, 256, 128, 2, 4))) == 0
    # H and I at most 4096 (two pipeline slots of 32 weight rows x K in shared memory)
    assert lib.moe_workspace_bytes(ctypes.byref(dims(8, 4096, 4096, 2, 4))) > 0
    assert lib.moe_workspace_bytes(ctypes.byref(dims(8, 4160, 128, 2, 4))) == 0
    assert lib.moe_workspace_bytes(ctypes.byref(dims(8, 256, 4160, 2, 4))) == 0


def _call(lib, d, ptr=16, ws_bytes=1 << 30):
    p = ctypes.c_void_p(ptr)
    return lib.moe_a16w4_mxfp4(ctypes.byref(d), p, p, p, p, p, p, p, p, ctypes.c_void_p(256), ws_bytes, None)


def test_argument_errors_are_host_side(lib):
    from mxfp4_weight_only_gb300 import MOE_PATH_PREFILL, MoeDims, dims

    assert _call(lib, MoeDims(8, 256, 128, 2, 4, 1, 0)) == -4  # unsupported activation: fail closed
    assert _call(lib, dims(8, 250, 128, 2, 4)) == -2  # H not a multiple of 64
    assert _call(lib, dims(8, 256, 128, 2, 4), ptr=0) == -1  # NULL pointers
    assert _call(lib, dims(8, 256, 128, 2, 4), ptr=8) == -3  # misaligned
    assert _call(lib, dims(8, 256, 128, 2, 4), ws_bytes=16) == -5  # workspace too small
    assert _call(lib, dims(8, 256, 128, 2, 0)) == 0  # T = 0: nothing to do
    # the tensor-core path needs H and I multiples of 512
    assert _call(lib, dims(8, 256, 128, 2, 4, MOE_PATH_PREFILL)) == -2
    n = lib.requant_mxfp4_to_int4g32(2, 4, 48, None, None, None, None, 8, None)
    assert n == -2  # K % 32
    assert lib.requant_mxfp4_to_int4g32(2, 4, 64, None, None, None, None, 8, None) == -1
    # the bounded-wait hook rejects a zero limit and out-of-range extra waiters
    assert lib.moe_set_wait_limit(0, 0) == -2
    assert lib.moe_set_wait_limit(1000, -1) == -2
    assert lib.moe_set_wait_limit(1000, 65) == -2
    assert lib.moe_noalloc_read_status(None, None) == -1


def test_router_errors_are_host_side(lib):
    p = ctypes.c_void_p(16)
    assert lib.moe_router_topk(p, 4, 1025, 8, 1, p, p, None) == -2  # more than 1024 experts
    assert lib.moe_router_topk(p, 4, 32, 65, 1, p, p, None) == -2  # top-k above 64
    assert lib.moe_router_topk(p, 4, 8, 9, 1, p, p, None) == -2  # top-k above the experts
    assert lib.moe_router_topk(p, 4, 32, 4, 2, p, p, None) == -2  # renormalize not 0 / 1
    assert lib.moe_router_topk(None, 4, 32, 4, 1, p, p, None) == -1
    assert lib.moe_router_topk(ctypes.c_void_p(18), 4, 32, 4, 1, p, p, None) == -3
    assert lib.moe_router_topk(None, 0, 32, 4, 1, None, None, None) == 0  # T = 0: nothing to do


def test_option_errors_are_host_side(lib):
    from mxfp4_weight_only_gb300 import MoeOptions, dims

    d = dims(8, 256, 128, 2, 4)
    p = ctypes.c_void_p(16)

    def call(opt):
        return lib.moe_a16w4_mxfp4_ex(ctypes.byref(d), p, p, p, p, p, p, p, ctypes.byref(opt), p,
                                      ctypes.c_void_p(256), 1 << 30, None)

    assert call(MoeOptions(None, None, None, 0, 2)) == -2  # router_weight_on_input not 0 / 1
    assert call(MoeOptions(None, None, 64, 0, 0)) == -2  # a map with no entries
    assert call(MoeOptions(None, None, 64, (1 << 20) + 1, 0)) == -2
    assert call(MoeOptions(17, None, None, 0, 0)) == -3  # bias not 2-byte aligned
    assert call(MoeOptions(None, None, 66, 8, 0)) == -3  # map not 4-byte aligned
    # activation quantisation: mode, FP8 scales, no router weight on the input
    assert call(MoeOptions(None, None, None, 0, 0, 3, 1.0, 1.0)) == -2
    assert call(MoeOptions(None, None, None, 0, 0, -1, 1.0, 1.0)) == -2
    for s13, s2 in ((0.0, 1.0), (1.0, -2.0), (float("nan"), 1.0), (1.0, float("inf"))):
        assert call(MoeOptions(None, None, None, 0, 0, 2, s13, s2)) == -2
    assert call(MoeOptions(None, None, None, 0, 1, 1, 1.0, 1.0)) == -2
    assert call(MoeOptions(None, None, None, 0, 1, 2, 0.5, 0.5)) == -2
    # swiglu_limit: finite and >= 0 (0 = off)
    for lim in (-1.0, float("nan"), float("inf")):
        assert call(MoeOptions(None, None, None, 0, 0, 0, 1.0, 1.0, lim)) == -2
    # not with int4 weights
    opt = MoeOptions(None, None, None, 0, 0, 1, 1.0, 1.0)
    assert lib.moe_a16w4_int4g32_ex(ctypes.byref(d), p, p, p, p, p, p, p, ctypes.byref(opt), p,
                                    ctypes.c_void_p(256), 1 << 30, None) == -2


def test_quantize_act_errors_are_host_side(lib):
    p = ctypes.c_void_p(16)
    assert lib.moe_quantize_act(0, p, 0, 4, 64, 1.0, p, p, None) == -2  # no quantisation mode
    assert lib.moe_quantize_act(3, p, 0, 4, 64, 1.0, p, p, None) == -2
    assert lib.moe_quantize_act(1, p, 2, 4, 64, 1.0, p, p, None) == -2  # dtype flag
    assert lib.moe_quantize_act(1, p, 0, 4, 48, 1.0, p, p, None) == -2  # K % 32
    assert lib.moe_quantize_act(1, p, 0, -1, 64, 1.0, p, p, None) == -2
    assert lib.moe_quantize_act(2, p, 0, 4, 64, 0.0, p, None, None) == -2  # FP8 scale
    assert lib.moe_quantize_act(2, p, 0, 4, 64, float("nan"), p, None, None) == -2
    assert lib.moe_quantize_act(1, p, 0, 4, 64, 1.0, p, None, None) == -1  # MX scales need an output
    assert lib.moe_quantize_act(1, None, 0, 4, 64, 1.0, p, p, None) == -1
    assert lib.moe_quantize_act(2, ctypes.c_void_p(8), 0, 4, 64, 1.0, p, None, None) == -3
    assert lib.moe_quantize_act(1, None, 0, 0, 64, 1.0, None, None, None) == 0  # no rows: nothing to do
