"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Integer outputs (routing, requantised codes and scales) must match bit for
bit; MoE outputs must satisfy the tolerance in tests/tolerance.py.  Small
cases are compared element by element in full; the full-size expert-parallel
shape is compared on sampled outputs that the oracle computes one by one.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import formats, moe, requant, route
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


def x_dev(x_bits):
    return torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)


def out_host(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def gaussian_problem(seed, E, H, I, T, topk, bias_std=None):
    g = synth.rng(seed)
    x = synth.activations_bf16(g, T, H)
    ids, w = synth.router_topk(g, T, E, topk, bias_std)
    w13, s13 = formats.quantize_mxfp4(synth.gaussian(g, (E, 2 * I, H), 0.02))
    w2, s2 = formats.quantize_mxfp4(synth.gaussian(g, (E, H, I), 0.02))
    return x, ids, w, w13, s13, w2, s2


def run_gpu(m, prob, path=0, kind="mxfp4"):
    x, ids, w, w13, s13, w2, s2 = prob
    fn = m.moe_a16w4_mxfp4 if kind == "mxfp4" else m.moe_a16w4_int4g32
    out = fn(x_dev(x), dev(ids), dev(w), dev(w13), dev(s13), dev(w2), dev(s2), path=path)
    torch.cuda.synchronize()
    return formats.bf16_to_f64(out_host(out))


# ----------------------------------------------------------------------------- routing


@pytest.mark.parametrize("T,topk,E,lo,hi", [(4, 2, 8, 0, 8), (1, 15, 112, 0, 112), (32, 15, 112, -3, 115),
                                            (4096, 15, 112, 0, 112), (3000, 7, 1024, -5, 1030), (0, 4, 8, 0, 8)])
def test_route_bitexact(mw, T, topk, E, lo, hi):
    g = np.random.default_rng(T + topk + E)
    ids = g.integers(lo, hi, size=(T, topk)).astype(np.int32)
    c, o, sp, pos = mw.moe_route(dev(ids), E)
    rc, ro, rsp, rpos = route.route(ids, E)
    assert np.array_equal(c.cpu().numpy(), rc)
    assert np.array_equal(o.cpu().numpy(), ro)
    assert np.array_equal(sp.cpu().numpy(), rsp)
    assert np.array_equal(pos.cpu().numpy(), rpos)


# ----------------------------------------------------------------------------- requantiser


def _requant_check(mw, w, sc, chunk=8):
    q, s = mw.requant_mxfp4_to_int4g32(dev(w), dev(sc), experts_per_chunk=chunk)
    torch.cuda.synchronize()
    rq, rs = requant.requant_mxfp4_to_int4g32(w, sc, chunk)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


@pytest.mark.parametrize("s_lo,s_hi", [(0, 12), (100, 140), (240, 252)])
def test_requant_bitexact_scale_ranges(mw, s_lo, s_hi):
    g = np.random.default_rng(s_lo + 7)
    E, N, K = 11, 48, 256
    w = g.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    w[0, :5] = 0  # all-zero groups
    w[1, 3, :16] = 0x88  # negative zeros only
    sc = g.integers(s_lo, s_hi + 1, size=(E, N, K // 32), dtype=np.uint8)
    _requant_check(mw, w, sc, chunk=8)


def test_requant_bitexact_gaussian_tiny(mw):
    g = synth.rng(0)
    w, s = formats.quantize_mxfp4(synth.gaussian(g, (8, 256, 256), 0.02))
    _requant_check(mw, w, s, chunk=3)


# ----------------------------------------------------------------------------- MoE, small problems in full


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_moe_tiny_config(mw, seed):
    S = synth.TINY
    prob = gaussian_problem(seed, S.E, S.H, S.I, S.T, S.topk)
    ref = moe.moe_forward(*prob)
    assert_moe_close(run_gpu(mw, prob), ref)


@pytest.mark.parametrize("E,H,I,T,topk", [(4, 192, 320, 37, 3), (16, 512, 256, 9, 4), (3, 64, 64, 1, 1),
                                          (1, 128, 192, 20, 1), (8, 1024, 512, 64, 8)])
def test_moe_ragged_shapes_decode(mw, E, H, I, T, topk):
    prob = gaussian_problem(E * 1000 + T, E, H, I, T, topk)
    ref = moe.moe_forward(*prob)
    assert_moe_close(run_gpu(mw, prob, path=1), ref)


@pytest.mark.parametrize("T,topk", [(16, 8), (43, 3), (129, 1)])
def test_moe_decode_grouping_limit(mw, T, topk):
    # the weight-streaming kernels group up to 128 pairs themselves and use the
    # routing kernel above that: P = 128 and P = 129 on either side, with a few
    # invalid ids, must both match the oracle
    E, H, I = 24, 512, 256
    prob = list(gaussian_problem(T * 31 + topk, E, H, I, T, topk))
    ids = prob[1].copy()
    ids.reshape(-1)[::17] = -1
    prob[1] = ids
    ref = moe.moe_forward(*prob)
    assert_moe_close(run_gpu(mw, prob, path=1), ref)


@pytest.mark.parametrize("E,H,I,T,topk", [(4, 4096, 256, 3, 2), (3, 256, 3840, 5, 2), (2, 4096, 4096, 2, 3)])
def test_moe_decode_two_launch_path(mw, E, H, I, T, topk):
    # H or I above 3584: the gate_up and down GEMMs run as two launches
    # (wider per-warp activation fragments) instead of the single fused one
    prob = gaussian_problem(E * 7 + H + I, E, H, I, T, topk)
    ref = moe.moe_forward(*prob)
    assert_moe_close(run_gpu(mw, prob, path=1), ref)


@pytest.mark.parametrize("fill", ["ones", "ramp", "zeros"])
def test_fused_decode_workspace_contents_irrelevant(mw, fill):
    # the fused decode kernel synchronises its CTAs through words in the
    # workspace; whatever the workspace held before, repeated calls on it must
    # all match the oracle and each other, also after moe_read_status clears it
    S = synth.TINY
    x, ids, w, w13, s13, w2, s2 = gaussian_problem(11, S.E, S.H, S.I, S.T, S.topk)
    ref = moe.moe_forward(x, ids, w, w13, s13, w2, s2)
    d = mw.dims(S.E, S.H, S.I, S.topk, S.T, 1)
    n = mw.moe_workspace_bytes(d)
    if fill == "ones":
        ws = torch.full((n,), 255, dtype=torch.uint8, device="cuda")
    elif fill == "ramp":
        ws = (torch.arange(n, device="cuda") % 251).to(torch.uint8)
    else:
        ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    ws[:4] = 0  # the status word reads what the memory held until first cleared
    args = (x_dev(x), dev(ids), dev(w), dev(w13), dev(s13), dev(w2), dev(s2))
    outs = []
    for i in range(6):
        if i == 3:
            assert mw.moe_read_status(d, ws) == 0
        out = mw.moe_a16w4_mxfp4(*args, workspace=ws, path=1)
        torch.cuda.synchronize()
        outs.append(out_host(out).copy())
    assert mw.moe_read_status(d, ws) == 0
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    assert_moe_close(formats.bf16_to_f64(outs[0]), ref)


def test_moe_invalid_and_duplicate_ids(mw):
    prob = list(gaussian_problem(5, 8, 256, 128, 6, 3))
    ids = prob[1]
    ids[0, 1] = -1
    ids[1, :] = [2, 2, 2]
    ids[2, :] = [-1, 8, 100]  # a token with no valid expert -> zero row
    ref = moe.moe_forward(*prob)
    got = run_gpu(mw, prob)
    assert np.all(got[2] == 0)
    assert_moe_close(got, ref)


def test_moe_int4_small(mw):
    x, ids, w, w13, s13, w2, s2 = gaussian_problem(3, 8, 256, 128, 7, 2)
    q13, f13 = requant.requant_mxfp4_to_int4g32(w13, s13)
    q2, f2 = requant.requant_mxfp4_to_int4g32(w2, s2)
    prob = (x, ids, w, q13, f13, q2, f2)
    ref = moe.moe_forward(*prob, kind="int4g32")
    assert_moe_close(run_gpu(mw, prob, kind="int4"), ref)


def test_workspace_status_clean(mw):
    S = synth.TINY
    x, ids, w, w13, s13, w2, s2 = gaussian_problem(0, S.E, S.H, S.I, S.T, S.topk)
    d = mw.dims(S.E, S.H, S.I, S.topk, S.T)
    ws = torch.zeros(mw.moe_workspace_bytes(d), dtype=torch.uint8, device="cuda")
    mw.moe_a16w4_mxfp4(x_dev(x), dev(ids), dev(w), dev(w13), dev(s13), dev(w2), dev(s2), workspace=ws)
    assert mw.moe_read_status(d, ws) == 0


def test_repeat_calls_identical(mw):
    prob = gaussian_problem(4, 16, 512, 256, 9, 4)
    a = run_gpu(mw, prob)
    b = run_gpu(mw, prob)
    assert np.array_equal(a, b)


# ----------------------------------------------------------------------------- full-size expert-parallel shape


@pytest.fixture(scope="module")
def k3_weights(mw):
    S = synth.k3(1)
    g = synth.rng(100)
    w13, s13 = synth.random_mxfp4_bytes(g, S.E, 2 * S.I, S.H)
    w2, s2 = synth.random_mxfp4_bytes(g, S.E, S.H, S.I)
    return (w13, s13, w2, s2), tuple(dev(a) for a in (w13, s13, w2, s2))


@pytest.mark.parametrize("T", [1, 4, 7, 16, 32])
def test_moe_k3_decode_sampled(mw, k3_weights, T):
    (w13, s13, w2, s2), dw = k3_weights
    S = synth.k3(T)
    g = synth.rng(200 + T)
    x = synth.activations_bf16(g, T, S.H)
    ids, w = synth.router_topk(g, T, S.E, S.topk)
    out = mw.moe_a16w4_mxfp4(x_dev(x), dev(ids), dev(w), *dw)
    torch.cuda.synchronize()
    got = formats.bf16_to_f64(out_host(out))
    toks = np.unique(np.array([0, T - 1, T // 2]))[:2 if T >= 16 else 3]
    cols = np.sort(g.choice(S.H, 96, replace=False))
    ref = moe.moe_forward_sampled(x, ids, w, w13, s13, w2, s2, toks, cols)
    assert_moe_close(got[np.ix_(toks, cols)], ref)


def test_requant_k3_all_experts_sampled(mw, k3_weights):
    (w13, s13, w2, s2), (dw13, ds13, dw2, ds2) = k3_weights
    q, s = mw.requant_mxfp4_to_int4g32(dw13, ds13, experts_per_chunk=8)
    torch.cuda.synchronize()
    for e in (0, 57, 111):
        rq, rs = requant.requant_mxfp4_to_int4g32(w13[e:e + 1], s13[e:e + 1])
        assert np.array_equal(q[e].cpu().numpy(), rq[0])
        assert np.array_equal(s[e].cpu().numpy().view(np.uint32), rs[0].view(np.uint32))


@pytest.mark.parametrize("T", [1, 7, 32])
def test_moe_k3_int4_sampled(mw, k3_weights, T):
    (w13, s13, w2, s2), (dw13, ds13, dw2, ds2) = k3_weights
    q13, f13 = mw.requant_mxfp4_to_int4g32(dw13, ds13)
    q2, f2 = mw.requant_mxfp4_to_int4g32(dw2, ds2)
    S = synth.k3(T)
    g = synth.rng(300 + T)
    x = synth.activations_bf16(g, T, S.H)
    ids, w = synth.router_topk(g, T, S.E, S.topk)
    out = mw.moe_a16w4_int4g32(x_dev(x), dev(ids), dev(w), q13, f13, q2, f2)
    torch.cuda.synchronize()
    got = formats.bf16_to_f64(out_host(out))
    toks = np.array([0]) if T == 1 else np.array([0, T - 1])
    cols = np.sort(g.choice(S.H, 64, replace=False))
    need = sorted({int(e) for t in toks for e in ids[t]})
    # the oracle requantises the experts it needs from the same MXFP4 bytes
    oq13 = np.zeros_like(w13[:1]).repeat(S.E, 0)
    of13 = np.zeros((S.E,) + s13.shape[1:], np.float32)
    oq2 = np.zeros_like(w2[:1]).repeat(S.E, 0)
    of2 = np.zeros((S.E,) + s2.shape[1:], np.float32)
    for e in need:
        a, b = requant.requant_mxfp4_to_int4g32(w13[e:e + 1], s13[e:e + 1])
        oq13[e], of13[e] = a[0], b[0]
        a, b = requant.requant_mxfp4_to_int4g32(w2[e:e + 1], s2[e:e + 1])
        oq2[e], of2[e] = a[0], b[0]
    ref = moe.moe_forward_sampled(x, ids, w, oq13, of13, oq2, of2, toks, cols, kind="int4g32")
    assert_moe_close(got[np.ix_(toks, cols)], ref)


# ----------------------------------------------------------------------------- tensor-core (prefill) path


@pytest.mark.parametrize("E,H,I,T,topk,bias", [(8, 512, 512, 200, 4, None), (4, 512, 1024, 300, 2, 2.0),
                                               (16, 1024, 512, 130, 6, 2.0)])
def test_moe_prefill_small(mw, E, H, I, T, topk, bias):
    prob = gaussian_problem(E * 7 + T, E, H, I, T, topk, bias)
    ref = moe.moe_forward(*prob)
    assert_moe_close(run_gpu(mw, prob, path=2), ref)


@pytest.mark.parametrize("E,H,I,T,topk,bias", [(8, 512, 512, 200, 4, None), (5, 1024, 512, 130, 3, 2.0)])
def test_moe_int4_prefill_small(mw, E, H, I, T, topk, bias):
    x, ids, w, w13, s13, w2, s2 = gaussian_problem(E * 11 + T, E, H, I, T, topk, bias)
    q13, f13 = requant.requant_mxfp4_to_int4g32(w13, s13)
    q2, f2 = requant.requant_mxfp4_to_int4g32(w2, s2)
    prob = (x, ids, w, q13, f13, q2, f2)
    ref = moe.moe_forward(*prob, kind="int4g32")
    assert_moe_close(run_gpu(mw, prob, path=2, kind="int4"), ref)


def test_moe_prefill_tile_boundaries(mw):
    # gate_up items hold up to 192 rows of one expert, down items 128: expert 0
    # gets 193 rows (192 + 1 and 128 + 65), expert 1 exactly 192 (one item;
    # 128 + 64), expert 2 129 (one item; 128 + 1), expert 3 385 (192 + 192 + 1;
    # 3 x 128 + 1), expert 4 17 (an MMA N of 32 with 15 idle columns), expert
    # 5 none; invalid ids in between
    E, H, I, topk = 6, 512, 512, 1
    counts = [193, 192, 129, 385, 17]
    ids = np.concatenate([np.full(c, e, np.int32) for e, c in enumerate(counts)] + [np.array([-1, 7], np.int32)])
    g = np.random.default_rng(11)
    ids = ids[g.permutation(ids.size)][:, None].astype(np.int32)
    T = ids.shape[0]
    prob = list(gaussian_problem(12, E, H, I, T, topk))
    prob[1] = ids
    prob[2] = g.uniform(0.1, 1.0, size=(T, 1)).astype(np.float32)
    ref = moe.moe_forward(*prob)
    got = run_gpu(mw, prob, path=2)
    assert_moe_close(got, ref)
    assert np.all(got[(ids[:, 0] < 0) | (ids[:, 0] >= E)] == 0)


def test_prefill_and_decode_paths_agree_with_oracle(mw):
    prob = gaussian_problem(21, 8, 512, 512, 96, 4)
    ref = moe.moe_forward(*prob)
    a = run_gpu(mw, prob, path=1)
    b = run_gpu(mw, prob, path=2)
    assert_moe_close(a, ref)
    assert_moe_close(b, ref)
    c = run_gpu(mw, prob, path=0)  # T >= 64: the automatic choice is the tensor-core path
    assert_moe_close(c, ref)  # the tensor-core combine adds in arrival order: equal within tolerance


def test_moe_k3_int4_prefill_sampled(mw, k3_weights):
    (w13, s13, w2, s2), (dw13, ds13, dw2, ds2) = k3_weights
    q13, f13 = mw.requant_mxfp4_to_int4g32(dw13, ds13)
    q2, f2 = mw.requant_mxfp4_to_int4g32(dw2, ds2)
    T = 1024
    S = synth.k3(T)
    g = synth.rng(410)
    x = synth.activations_bf16(g, T, S.H)
    ids, w = synth.router_topk(g, T, S.E, S.topk, expert_bias_std=2.0)
    out = mw.moe_a16w4_int4g32(x_dev(x), dev(ids), dev(w), q13, f13, q2, f2)  # T >= 64: tensor-core path
    torch.cuda.synchronize()
    got = formats.bf16_to_f64(out_host(out))
    toks = np.array([0, T - 1])
    cols = np.sort(g.choice(S.H, 64, replace=False))
    need = sorted({int(e) for t in toks for e in ids[t]})
    oq13 = np.zeros_like(w13[:1]).repeat(S.E, 0)
    of13 = np.zeros((S.E,) + s13.shape[1:], np.float32)
    oq2 = np.zeros_like(w2[:1]).repeat(S.E, 0)
    of2 = np.zeros((S.E,) + s2.shape[1:], np.float32)
    for e in need:
        a, b = requant.requant_mxfp4_to_int4g32(w13[e:e + 1], s13[e:e + 1])
        oq13[e], of13[e] = a[0], b[0]
        a, b = requant.requant_mxfp4_to_int4g32(w2[e:e + 1], s2[e:e + 1])
        oq2[e], of2[e] = a[0], b[0]
    ref = moe.moe_forward_sampled(x, ids, w, oq13, of13, oq2, of2, toks, cols, kind="int4g32")
    assert_moe_close(got[np.ix_(toks, cols)], ref)
    assert np.isfinite(got).all()


def test_moe_k3_prefill_sampled(mw, k3_weights):
    (w13, s13, w2, s2), dw = k3_weights
    T = 4096
    S = synth.k3(T)
    g = synth.rng(400)
    x = synth.activations_bf16(g, T, S.H)
    ids, w = synth.router_topk(g, T, S.E, S.topk, expert_bias_std=2.0)
    out = mw.moe_a16w4_mxfp4(x_dev(x), dev(ids), dev(w), *dw)
    torch.cuda.synchronize()
    got = formats.bf16_to_f64(out_host(out))
    toks = np.array([0, 2047, 4095])
    cols = np.sort(g.choice(S.H, 96, replace=False))
    ref = moe.moe_forward_sampled(x, ids, w, w13, s13, w2, s2, toks, cols)
    assert_moe_close(got[np.ix_(toks, cols)], ref)
    assert np.isfinite(got).all()
