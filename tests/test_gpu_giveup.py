"""The give-up path of the kernels' bounded waits, run on the GPU without a fault.

The fused decode kernel's CTAs wait for one another's gate_up results.  The
library's wait hook (moe_set_wait_limit) gives the next call a 1 ms limit and
makes that wait expect one CTA more than the grid has, so the real wait code
runs out: the kernel must record MOE_STATUS_WAIT_TIMEOUT, stop its pipeline
and return, and the workspace must serve the next call correctly, whether or
not the status was read (and cleared) in between.
"""

import ctypes
import time

import numpy as np
import pytest
import torch

import synth
from oracle import formats, moe
from tests.tolerance import assert_moe_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mw():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mxfp4_weight_only_gb300 import build

    build.build()
    import mxfp4_weight_only_gb300 as m

    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def tiny_problem(seed):
    S = synth.TINY
    g = synth.rng(seed)
    x = synth.activations_bf16(g, S.T, S.H)
    ids, w = synth.router_topk(g, S.T, S.E, S.topk)
    w13, s13 = formats.quantize_mxfp4(synth.gaussian(g, (S.E, 2 * S.I, S.H), 0.02))
    w2, s2 = formats.quantize_mxfp4(synth.gaussian(g, (S.E, S.H, S.I), 0.02))
    return x, ids, w, w13, s13, w2, s2


def call(mw, prob, ws):
    x, ids, w, w13, s13, w2, s2 = prob
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    out = mw.moe_a16w4_mxfp4(xd, dev(ids), dev(w), dev(w13), dev(s13), dev(w2), dev(s2), workspace=ws,
                             path=mw.MOE_PATH_DECODE)
    torch.cuda.synchronize()
    return formats.bf16_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))


def force_give_up(mw):
    lib = mw._native.load()
    assert lib.moe_set_wait_limit(ctypes.c_uint64(1_000_000), 1) == 0  # 1 ms, one CTA that never comes


@pytest.mark.parametrize("read_between", [True, False])
def test_fused_decode_wait_gives_up_then_workspace_recovers(mw, read_between):
    S = synth.TINY
    d = mw.dims(S.E, S.H, S.I, S.topk, S.T, mw.MOE_PATH_DECODE)
    ws = torch.zeros(mw.moe_workspace_bytes(d), dtype=torch.uint8, device="cuda")
    prob = tiny_problem(3)
    ref = moe.moe_forward(*prob)
    assert_moe_close(call(mw, prob, ws), ref)
    assert mw.moe_read_status(d, ws) == 0

    force_give_up(mw)
    t0 = time.perf_counter()
    call(mw, prob, ws)  # output invalid by contract
    assert time.perf_counter() - t0 < 1.5  # the 1 ms limit, not the 2 s default, ended the waits
    if read_between:
        assert mw.moe_read_status(d, ws) == mw.MOE_STATUS_WAIT_TIMEOUT
    # the next calls on the same workspace are correct
    prob2 = tiny_problem(4)
    ref2 = moe.moe_forward(*prob2)
    for _ in range(2):
        assert_moe_close(call(mw, prob2, ws), ref2)
    expect = 0 if read_between else mw.MOE_STATUS_WAIT_TIMEOUT  # the bit stays until read
    assert mw.moe_read_status(d, ws) == expect
    assert mw.moe_read_status(d, ws) == 0


def test_wait_hook_applies_to_one_call_only(mw):
    S = synth.TINY
    d = mw.dims(S.E, S.H, S.I, S.topk, S.T, mw.MOE_PATH_DECODE)
    ws = torch.zeros(mw.moe_workspace_bytes(d), dtype=torch.uint8, device="cuda")
    prob = tiny_problem(5)
    force_give_up(mw)
    call(mw, prob, ws)
    assert mw.moe_read_status(d, ws) == mw.MOE_STATUS_WAIT_TIMEOUT
    assert_moe_close(call(mw, prob, ws), moe.moe_forward(*prob))
    assert mw.moe_read_status(d, ws) == 0
