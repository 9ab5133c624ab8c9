"""The allocation-free entry point (moe_a16w4_mxfp4_noalloc) against the regular one.

Callers that cannot allocate device memory when they run the layer use the
variant that keeps its scratch in a fixed device array inside the library.
This test calls both entry points through the C ABI on the same inputs, twice
in a row (the array keeps the previous call's contents), and requires the
variant's output to match the regular entry point's within the MoE tolerance.
It lives in its own file, collected last, so a failure here cannot stop the
rest of the GPU suite from running first.
"""

import ctypes

import numpy as np
import pytest
import torch

import synth
from oracle import formats
from tests.tolerance import assert_moe_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mxfp4_weight_only_gb300 import _native, build

    build.build()
    lib = _native.load()
    fn = lib.moe_a16w4_mxfp4_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(_native.MoeDims)] + [ctypes.c_void_p] * 9
    return lib


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _problem(seed, E, H, I, T, topk):
    g = synth.rng(seed)
    x = synth.activations_bf16(g, T, H)
    ids, w = synth.router_topk(g, T, E, topk)
    if E * I * H <= 1 << 24:
        w13, s13 = formats.quantize_mxfp4(synth.gaussian(g, (E, 2 * I, H), 0.02))
        w2, s2 = formats.quantize_mxfp4(synth.gaussian(g, (E, H, I), 0.02))
    else:  # full-size expert set: MXFP4 bytes drawn directly
        w13, s13 = synth.random_mxfp4_bytes(g, E, 2 * I, H)
        w2, s2 = synth.random_mxfp4_bytes(g, E, H, I)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    return (E, H, I, T, topk), (xd, dev(ids), dev(w), dev(w13), dev(s13), dev(w2), dev(s2))


def _regular(lib, shape, t):
    from mxfp4_weight_only_gb300 import _native

    E, H, I, T, topk = shape
    d = _native.MoeDims(E, H, I, topk, T, 0, 1)
    ws = torch.empty(lib.moe_workspace_bytes(ctypes.byref(d)), dtype=torch.uint8, device="cuda")
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    rc = lib.moe_a16w4_mxfp4(ctypes.byref(d), *[_p(a) for a in t], _p(out), _p(ws), ws.numel(),
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    return out


def _noalloc(lib, shape, t):
    from mxfp4_weight_only_gb300 import _native

    E, H, I, T, topk = shape
    d = _native.MoeDims(E, H, I, topk, T, 0, 0)
    out = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = lib.moe_a16w4_mxfp4_noalloc(ctypes.byref(d), *[_p(a) for a in t], _p(out),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, rc
    return out


def _noalloc_status(lib):
    v = ctypes.c_uint32(0xFFFFFFFF)
    rc = lib.moe_noalloc_read_status(ctypes.byref(v), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    return v.value


def _f64(t):
    return formats.bf16_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))


@pytest.mark.parametrize("shape_seed", [(8, 256, 128, 4, 2, 0), (112, 3584, 3072, 7, 15, 1)])
def test_noalloc_matches_regular_entry_point_twice(lib, shape_seed):
    E, H, I, T, topk, seed = shape_seed
    shape, a = _problem(seed, E, H, I, T, topk)
    ref = _f64(_regular(lib, shape, a))
    shape2, b = _problem(seed + 10, E, H, I, T, topk)
    ref2 = _f64(_regular(lib, shape2, b))
    # two calls in a row on different inputs: the second sees the first's leftovers
    got = _f64(_noalloc(lib, shape, a))
    got2 = _f64(_noalloc(lib, shape2, b))
    torch.cuda.synchronize()
    assert_moe_close(got, ref)
    assert_moe_close(got2, ref2)
    assert _noalloc_status(lib) == 0


def test_noalloc_wait_give_up_is_reported_and_cleared(lib):
    # a bounded wait that runs out (1 ms limit, one CTA expected beyond the
    # grid) is recorded in the array's status word; reading it clears the word
    # and the synchronisation words, and the next call is correct again
    shape, a = _problem(2, 8, 256, 128, 4, 2)
    ref = _f64(_regular(lib, shape, a))
    assert lib.moe_set_wait_limit(ctypes.c_uint64(1_000_000), 1) == 0
    _noalloc(lib, shape, a)
    torch.cuda.synchronize()
    assert _noalloc_status(lib) == 1  # MOE_STATUS_WAIT_TIMEOUT
    got = _f64(_noalloc(lib, shape, a))
    assert_moe_close(got, ref)
    assert _noalloc_status(lib) == 0


def test_noalloc_rejects_oversized_problem(lib):
    from mxfp4_weight_only_gb300 import _native

    d = _native.MoeDims(112, 3584, 3072, 15, 4096, 0, 0)
    null = ctypes.c_void_p(16)
    rc = lib.moe_a16w4_mxfp4_noalloc(ctypes.byref(d), *([null] * 8), null)
    assert rc == -5  # MOE_ERR_WORKSPACE: beyond the fixed scratch size
