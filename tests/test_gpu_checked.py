"""The bounds-checked build (``libmoe_a16w4_check.so``: the same kernels
compiled with -DMOE_CHECK), the stand-in for a memory checker.

Its kernels check every index they derive from the grouping (expert, pair,
token, row, tile) against its buffer and every E8M0 weight-scale byte they
read; a bad index is recorded in the status word and replaced by 0, so no
access leaves its buffer.  Every path runs here on small problems through the
checked build: the outputs match the oracle and the status word stays 0.
Weight scales holding the E8M0 NaN byte (255, outside the layer's contract)
are reported with MOE_STATUS_NAN_SCALE.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import formats, moe, requant
from tests.tolerance import assert_moe_close

pytestmark = pytest.mark.gpu

PATH_DECODE, PATH_PREFILL = 1, 2


@pytest.fixture(scope="module")
def mw():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mxfp4_weight_only_gb300 import build

    build.build()
    import mxfp4_weight_only_gb300 as m

    m.use_checked(True)
    yield m
    m.use_checked(False)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def problem(seed, E, H, I, T, topk):
    g = synth.rng(seed)
    x = synth.activations_bf16(g, T, H)
    ids, w = synth.router_topk(g, T, E, topk)
    ids[0, -1] = -1  # an invalid id: contributes nothing, not an index error
    w13, s13 = formats.quantize_mxfp4(synth.gaussian(g, (E, 2 * I, H), 0.02))
    w2, s2 = formats.quantize_mxfp4(synth.gaussian(g, (E, H, I), 0.02))
    return x, ids, w, w13, s13, w2, s2


def run(mw, prob, path, kind="mxfp4", **kw):
    x, ids, w, a, b, c, d = prob
    T, H = x.shape
    E, two_i = a.shape[0], a.shape[1]
    dims = mw.dims(E, H, two_i // 2, ids.shape[1], T, path)
    ws = torch.zeros(mw.moe_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    fn = mw.moe_a16w4_mxfp4 if kind == "mxfp4" else mw.moe_a16w4_int4g32
    out = fn(xd, dev(ids), dev(w), dev(a), dev(b), dev(c), dev(d), path=path, workspace=ws, **kw)
    status = mw.moe_read_status(dims, ws)
    return formats.bf16_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16)), status


def test_the_checked_library_is_the_one_called(mw):
    from mxfp4_weight_only_gb300 import _native, build

    assert _native.load() is _native.load(checked=True)
    assert _native.load()._name == build.lib_path(checked=True)


@pytest.mark.parametrize("path,E,H,I,T,topk", [
    (PATH_DECODE, 8, 512, 256, 3, 2),     # fused, grouping by one warp
    (PATH_DECODE, 8, 512, 256, 20, 4),    # fused, grouping by the CTA
    (PATH_DECODE, 8, 512, 256, 70, 4),    # routing kernel
    (PATH_DECODE, 6, 4096, 256, 5, 2),    # two launches
    (PATH_PREFILL, 8, 512, 512, 300, 3),  # tensor-core kernels
])
def test_every_path_clean_and_correct(mw, path, E, H, I, T, topk):
    prob = problem(10 + T, E, H, I, T, topk)
    got, status = run(mw, prob, path)
    assert status == 0
    assert_moe_close(got, moe.moe_forward(*prob))


@pytest.mark.parametrize("path,T", [(PATH_DECODE, 9), (PATH_PREFILL, 200)])
def test_int4_clean_and_correct(mw, path, T):
    x, ids, w, w13, s13, w2, s2 = problem(40 + T, 8, 512, 512, T, 2)
    q13, f13 = requant.requant_mxfp4_to_int4g32(w13, s13)
    q2, f2 = requant.requant_mxfp4_to_int4g32(w2, s2)
    prob = (x, ids, w, q13, f13, q2, f2)
    got, status = run(mw, prob, path, kind="int4")
    assert status == 0
    assert_moe_close(got, moe.moe_forward(*prob, kind="int4g32"))


def test_options_clean(mw):
    E, H, I, T, topk, G = 6, 512, 512, 7, 3, 16
    prob = problem(77, E, H, I, T, topk)
    g = synth.rng(78)
    emap = np.full(G, -1, np.int32)
    emap[g.choice(G, E, replace=False)] = np.arange(E, dtype=np.int32)
    gids = g.integers(0, G, size=(T, topk)).astype(np.int32)
    x, _, w, w13, s13, w2, s2 = prob
    prob = (x, gids, w, w13, s13, w2, s2)
    for path in (PATH_DECODE, PATH_PREFILL):
        got, status = run(mw, prob, path, expert_map=dev(emap), act_quant="fp8", w13_input_scale=0.05,
                          w2_input_scale=0.01)
        assert status == 0
        assert np.isfinite(got).all()


@pytest.mark.parametrize("path,T", [(PATH_DECODE, 4), (PATH_PREFILL, 200)])
@pytest.mark.parametrize("which", ["w13", "w2"])
def test_nan_scale_byte_is_reported(mw, path, T, which):
    x, ids, w, w13, s13, w2, s2 = problem(90 + T, 4, 512, 512, T, 2)
    ids[:] = 1  # every pair on expert 1
    s13, s2 = s13.copy(), s2.copy()
    (s13 if which == "w13" else s2)[1, 3, 0] = 255
    _, status = run(mw, (x, ids, w, w13, s13, w2, s2), path)
    assert status & mw.MOE_STATUS_NAN_SCALE
    assert not status & mw.MOE_STATUS_BAD_INDEX
