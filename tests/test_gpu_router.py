"""GPU parity of the top-k router (moe_router_topk) against the oracle.

Ids must match bit for bit (the kernel selects by logit, which orders the
experts exactly as their softmax probabilities do; ties go to the lower id);
weights within a relative 1e-5 of the float64 oracle (float32 exp and one
IEEE division per weight).  The routed ids then feed the MoE layer, which is
compared with the oracle on the same ids.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import formats, moe, route
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


def check(mw, logits, topk, renorm=True):
    ids, w = mw.moe_router_topk(torch.from_numpy(logits).cuda(), topk, renormalize=renorm)
    torch.cuda.synchronize()
    rid, rw = route.router_topk(logits, topk, renormalize=renorm)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=1e-5, atol=0)
    return ids, w


@pytest.mark.parametrize("T,G,topk", [(1, 896, 15), (37, 112, 15), (5, 1024, 64), (9, 64, 64), (3, 7, 1),
                                      (0, 112, 15)])
def test_router_matches_oracle(mw, T, G, topk):
    g = np.random.default_rng(T * 7 + G)
    logits = g.standard_normal((T, G)).astype(np.float32)
    for renorm in (True, False):
        check(mw, logits, topk, renorm)


def test_router_ties_and_infinities(mw):
    g = np.random.default_rng(3)
    logits = g.standard_normal((4, 100)).astype(np.float32)
    logits[0, [5, 40, 70, 99]] = 3.0                # four-way tie at the top
    logits[1, :] = 0.5                               # every logit equal
    logits[2, 50:] = -np.inf                         # masked experts, top-k reaches into them
    logits[3, [0, 31, 32, 63, 64, 95]] = 9.0         # ties across lanes and register slots
    check(mw, logits, 8)
    check(mw, logits[:3], 60)  # row 2: the selection reaches into the -inf logits (weight 0)


def test_router_then_layer(mw):
    # router output feeding the layer through an expert map (896 global
    # experts, 112 of them on this GPU)
    T, G, E, H, I, topk = 6, 896, 16, 256, 128, 15
    g = np.random.default_rng(9)
    logits = g.standard_normal((T, G)).astype(np.float32)
    ids, w = check(mw, logits, topk)
    emap = np.full(G, -1, np.int32)
    emap[g.choice(G, E, replace=False)] = np.arange(E)
    x = synth.activations_bf16(g, T, H)
    w13, s13 = formats.quantize_mxfp4(synth.gaussian(g, (E, 2 * I, H), 0.02))
    w2, s2 = formats.quantize_mxfp4(synth.gaussian(g, (E, H, I), 0.02))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    out = mw.moe_a16w4_mxfp4(xd, ids, w, dev(w13), dev(s13), dev(w2), dev(s2), expert_map=dev(emap))
    torch.cuda.synchronize()
    got = formats.bf16_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
    ref = moe.moe_forward(x, ids.cpu().numpy(), w.cpu().numpy(), w13, s13, w2, s2, expert_map=emap)
    assert_moe_close(got, ref)
