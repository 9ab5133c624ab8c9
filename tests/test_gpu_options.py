"""GPU parity of the layer's optional inputs against the oracle.

Expert biases (``w13_bias`` / ``w2_bias``), the router weight applied on the
input, and the expert-parallel ``expert_map`` (global ids mapped to this
GPU's experts or -1): the Mxfp4MoEMethod page's ``create_weights`` /
``get_fused_moe_quant_config`` (biases) and ``apply`` (the other two).  Each
runs on the weight-streaming path (the fused kernel with in-kernel grouping,
the routing kernel above 128 pairs, the two-launch kernels for H above 3584)
and the tensor-core path, MXFP4 and int4.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import formats, moe, requant
from tests.tolerance import assert_moe_close

pytestmark = pytest.mark.gpu

DECODE, PREFILL = 1, 2


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


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def problem(seed, E, H, I, T, topk, G=None):
    """Gaussian MXFP4 experts, biases, and top-k ids; with G, ids are global
    ids in [-1, G] (some outside the map) and a map sends a random E of the G
    global experts to local ids, the rest to -1."""
    g = synth.rng(seed)
    x = synth.activations_bf16(g, T, H)
    if G is None:
        ids, w = synth.router_topk(g, T, E, topk)
        emap = None
    else:
        ids, w = synth.router_topk(g, T, G, topk)
        ids.reshape(-1)[::13] = G  # outside the map
        emap = np.full(G, -1, np.int32)
        emap[g.choice(G, E, replace=False)] = g.permutation(E)
    w13, s13 = formats.quantize_mxfp4(synth.gaussian(g, (E, 2 * I, H), 0.02))
    w2, s2 = formats.quantize_mxfp4(synth.gaussian(g, (E, H, I), 0.02))
    b13 = synth.bf16_bits_from_f32(synth.gaussian(g, (E, 2 * I), 0.5))
    b2 = synth.bf16_bits_from_f32(synth.gaussian(g, (E, H), 0.05))
    return x, ids, w, w13, s13, w2, s2, b13, b2, emap


def run(mw, prob, path, bias, rwi, use_map, kind="mxfp4", limit=None):
    x, ids, w, w13, s13, w2, s2, b13, b2, emap = prob
    if kind == "int4":
        w13, s13 = requant.requant_mxfp4_to_int4g32(w13, s13)
        w2, s2 = requant.requant_mxfp4_to_int4g32(w2, s2)
    kw = dict(router_weight_on_input=rwi, swiglu_limit=limit)
    okw = dict(router_weight_on_input=rwi, kind="mxfp4" if kind == "mxfp4" else "int4g32", swiglu_limit=limit)
    if bias:
        kw.update(w13_bias=bf16_dev(b13), w2_bias=bf16_dev(b2))
        okw.update(b13=b13, b2=b2)
    if use_map:
        kw.update(expert_map=dev(emap))
        okw.update(expert_map=emap)
    fn = mw.moe_a16w4_mxfp4 if kind == "mxfp4" else mw.moe_a16w4_int4g32
    out = fn(bf16_dev(x), dev(ids), dev(w), dev(w13), dev(s13), dev(w2), dev(s2), path=path, **kw)
    torch.cuda.synchronize()
    got = formats.bf16_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
    ref = moe.moe_forward(x, ids, w, w13, s13, w2, s2, **okw)
    return got, ref


CASES = [  # (path, E, H, I, T, topk): fused + in-kernel grouping, routing kernel, two launches, tensor cores
    (DECODE, 8, 512, 256, 9, 4),
    (DECODE, 12, 512, 256, 40, 4),
    (DECODE, 4, 4096, 256, 3, 2),
    (PREFILL, 8, 512, 512, 150, 3),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("bias,rwi", [(True, False), (False, True), (True, True)])
def test_bias_and_router_weight_on_input(mw, case, bias, rwi):
    path, E, H, I, T, topk = case
    prob = problem(E * 100 + T + 7 * bias + 3 * rwi, E, H, I, T, topk)
    assert_moe_close(*run(mw, prob, path, bias, rwi, False))


@pytest.mark.parametrize("case", CASES)
def test_expert_map(mw, case):
    path, E, H, I, T, topk = case
    prob = problem(E * 31 + T, E, H, I, T, topk, G=3 * E)
    got, ref = run(mw, prob, path, False, False, True)
    assert_moe_close(got, ref)
    # tokens none of whose experts is local come out as zeros
    x, ids, *_, emap = prob
    local = np.where((ids >= 0) & (ids < emap.size), emap[np.clip(ids, 0, emap.size - 1)], -1)
    none = ~(local >= 0).any(axis=1)
    assert np.all(got[none] == 0)


@pytest.mark.parametrize("path", [DECODE, PREFILL])
def test_all_options_together_int4(mw, path):
    E, H, I, T, topk = 6, 512, 512, (5 if path == DECODE else 140), 3
    prob = problem(77 + T, E, H, I, T, topk, G=2 * E)
    assert_moe_close(*run(mw, prob, path, True, True, True, kind="int4"))


def test_all_options_together_mxfp4_fused(mw):
    prob = problem(78, 8, 512, 256, 6, 4, G=20)
    assert_moe_close(*run(mw, prob, DECODE, True, True, True))


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("kind", ["mxfp4", "int4"])
def test_swiglu_limit(mw, case, kind):
    # the gate_up outputs (bias included) clamped to [-0.4, 0.4]: about half of
    # them are clamped here
    path, E, H, I, T, topk = case
    prob = problem(E * 17 + T, E, H, I, T, topk)
    got, ref = run(mw, prob, path, True, False, False, kind=kind, limit=0.4)
    assert_moe_close(got, ref)
    plain = run(mw, prob, path, True, False, False, kind=kind)[1]
    assert not np.allclose(ref, plain, rtol=1e-2)  # the clamp changes the layer

