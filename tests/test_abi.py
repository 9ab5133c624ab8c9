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


def test_version_and_error_strings(lib):
    assert lib.moe_abi_version() == 100
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
