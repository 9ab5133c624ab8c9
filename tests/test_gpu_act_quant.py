"""GPU parity of the W4A4 / W4A8 activation quantisation (vLLM PR #39136
schemes ``w_mxfp4_a_mxfp4`` and ``w_mxfp4_a_fp8``) against the CPU oracle.

* moe_quantize_act: codes and MX scale bytes bit-exact against
  ``oracle.actquant`` on bf16 and float32 rows, including E2M1 / e4m3 ties,
  saturation, negative zeros, all-zero and tiny blocks.
* The layer with quantised activations, weight-streaming and tensor-core
  kernels, fused and two-launch decode, with and without biases:
  - "exact-h" inputs (small integers times E2M1 weights whose scales keep
    every partial sum exact in float32, power-of-two FP8 input scales), where
    the gate_up result has no rounding error in any summation order, so both
    sides quantise the same intermediate up to the SiLU's rounding: the
    ordinary tolerance plus an allowance that is zero except where a few
    single intermediate values sit on a decision (at most 5e-2 of the RMS)
    -- tests/actquant_allowance.py;
  - Gaussian inputs, with the allowance from a probabilistic bound on the
    kernels' float32 error;
  - the same outputs compared with the A16W4 oracle fail the tolerance, so
    the quantisation is really applied.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import actquant, formats, moe
from tests.actquant_allowance import stage2_allowance
from tests.tolerance import ATOL_RMS, RTOL, moe_tolerance_report

pytestmark = pytest.mark.gpu

PATH_DECODE, PATH_PREFILL = 1, 2


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


# ------------------------------------------------------------------ the quantiser


def _edge_rows(K=256, seed=0):
    """Rows whose blocks hit the quantisers' decisions: E2M1 ties (v / X at
    0.25, 0.75, 1.25, ..., 5), saturation, -0.0, zero and tiny blocks."""
    g = np.random.default_rng(seed)
    rows = []
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 0.0])
    for sb in (1, 60, 120, 127, 133, 200, 250):
        X = 2.0 ** (sb - 127)
        blk = np.concatenate([ties, -ties, g.uniform(-6, 6, 32 - 2 * ties.size)]) * X
        blk[0] = 6.0 * X  # sets the block's scale to sb
        rows.append(blk)
    rows.append(np.full(32, -0.0))
    rows.append(np.zeros(32))
    rows.append(np.full(32, 2.0 ** -133))
    flat = np.concatenate(rows)
    flat = np.concatenate([flat, g.standard_normal(K - flat.size % K)])
    return flat.reshape(-1, K)


def _rows(kind, seed):
    g = np.random.default_rng(seed)
    rand = g.standard_normal((96, 256)) * np.exp2(g.integers(-40, 40, size=(96, 8)).repeat(32, 1))
    v = np.concatenate([_edge_rows(seed=seed), rand]).astype(np.float32)
    if kind == "bf16":
        bits = synth.bf16_bits_from_f32(v)
        return bf16_dev(bits), formats.bf16_to_f64(bits)
    return dev(v), v.astype(np.float64)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_quantize_act_mxfp4_bitexact(mw, dtype):
    xd, v = _rows(dtype, 1)
    q, qs = mw.moe_quantize_act(xd, "mxfp4")
    torch.cuda.synchronize()
    rq, rs = actquant.quantize_mxfp4_act(v)
    assert np.array_equal(qs.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("scale", [1.0, 0.25, 0.0123, 37.0])
def test_quantize_act_fp8_bitexact(mw, dtype, scale):
    xd, v = _rows(dtype, 2)
    if dtype == "f32":
        # the rows times the scale (finite inputs: rows that would overflow
        # float32 are dropped); quotients beyond 448 saturate
        keep = np.abs(v).max(1) * scale < 1e38
        v = (v[keep] * np.float32(scale)).astype(np.float32)
        xd = dev(v)
        v = v.astype(np.float64)
    q, _ = mw.moe_quantize_act(xd, "fp8", scale)
    torch.cuda.synchronize()
    rc, _ = actquant.quantize_fp8_act(v, scale)
    assert np.array_equal(q.cpu().numpy(), rc)


def test_quantize_act_fp8_ties_and_saturation(mw):
    vals = torch.tensor([0, 1, 2, 3, 0x7E, 0x80, 0xFE] + list(range(8, 0x7E)), dtype=torch.uint8)
    grid = np.unique(np.abs(vals.view(torch.float8_e4m3fn).double().numpy()))
    mids = (grid[:-1] + grid[1:]) / 2
    v = np.concatenate([grid, mids, -mids, [448.0, 464.0, 500.0, -1e6, -0.0, 2.0 ** -10, 3 * 2.0 ** -10]])
    v = np.concatenate([v, np.zeros((-v.size) % 32)]).astype(np.float32).reshape(-1, 32)
    q, _ = mw.moe_quantize_act(dev(v), "fp8", 0.5)  # power of two: v / 0.5 exact
    torch.cuda.synchronize()
    rc, _ = actquant.quantize_fp8_act(v.astype(np.float64), 0.5)
    assert np.array_equal(q.cpu().numpy(), rc)


@pytest.mark.parametrize("scale", [0.0123, 37.0, 3.3e-5, 1e-24, 1e23, 1.7e30])
def test_quantize_act_fp8_near_midpoints(mw, scale):
    # v = fl32(m * scale) and its float32 neighbours, m every e4m3 midpoint:
    # quotients v / scale within a few ulps of a rounding decision (the
    # kernels' multiply-by-reciprocal path must hand these to the division)
    vals = torch.arange(0, 0x7F, dtype=torch.uint8)
    grid = np.unique(vals.view(torch.float8_e4m3fn).double().numpy())
    mids = ((grid[:-1] + grid[1:]) / 2 * scale).astype(np.float32)
    near = [mids]
    for k in (1, 2, 3):
        near.append(np.nextafter(near[-1], np.float32(np.inf)))
    down = [mids]
    for k in (1, 2, 3):
        down.append(np.nextafter(down[-1], np.float32(0)))
    v = np.concatenate(near + down[1:])
    v = np.concatenate([v, -v])
    v = np.concatenate([v, np.zeros((-v.size) % 32, np.float32)]).reshape(-1, 32)
    q, _ = mw.moe_quantize_act(dev(v), "fp8", scale)
    torch.cuda.synchronize()
    rc, _ = actquant.quantize_fp8_act(v.astype(np.float64), scale)
    assert np.array_equal(q.cpu().numpy(), rc)


# ------------------------------------------------------------------ the layer


def exact_problem(seed, E, H, I, T, topk):
    """Integer x in [-8, 8], every E2M1 code, weight scales 2^-10 .. 2^-6:
    products are multiples of 2^-12 and every partial sum of h stays below
    K * 8 * 6 * 2^-6 <= 2^11.5 (K <= 4096 would need 2^23.5 units: exact)."""
    g = synth.rng(seed)
    x = synth.bf16_bits_from_f32(g.integers(-8, 9, size=(T, H)).astype(np.float32))
    ids, w = synth.router_topk(g, T, E, topk)
    w13 = g.integers(0, 256, size=(E, 2 * I, H // 2), dtype=np.uint8)
    w2 = g.integers(0, 256, size=(E, H, I // 2), dtype=np.uint8)
    s13 = g.integers(117, 122, size=(E, 2 * I, H // 32), dtype=np.uint8)
    s2 = g.integers(117, 122, size=(E, H, I // 32), dtype=np.uint8)
    return x, ids, w, w13, s13, w2, s2


def gaussian_problem(seed, E, H, I, T, topk):
    g = synth.rng(seed)
    x = synth.activations_bf16(g, T, H)
    ids, w = synth.router_topk(g, T, E, topk)
    w13, s13 = formats.quantize_mxfp4(synth.gaussian(g, (E, 2 * I, H), 0.02))
    w2, s2 = formats.quantize_mxfp4(synth.gaussian(g, (E, H, I), 0.02))
    return x, ids, w, w13, s13, w2, s2


def run(mw, prob, path, mode, si13, si2, **kw):
    x, ids, w, a, b, c, d = prob
    out = mw.moe_a16w4_mxfp4(bf16_dev(x), dev(ids), dev(w), dev(a), dev(b), dev(c), dev(d), path=path,
                             act_quant=mode, w13_input_scale=si13, w2_input_scale=si2, **kw)
    torch.cuda.synchronize()
    return formats.bf16_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))


def assert_close_with_allowance(got, ref, allow):
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = np.abs(got - ref)
    bad = ~(err <= ATOL_RMS * rms + RTOL * np.abs(ref) + allow)
    assert not bad.any(), (f"{int(bad.sum())} outside tolerance + allowance; first {np.argwhere(bad)[0]}, "
                           f"max err / rms {err.max() / rms:.3g}, allowance > 0 on {(allow > 0).mean():.3g}")


def check_layer(mw, prob, path, mode, si13, si2, h_exact, b13=None, b2=None):
    kw = {}
    if b13 is not None:
        kw = {"w13_bias": bf16_dev(b13), "w2_bias": bf16_dev(b2)}
    got = run(mw, prob, path, mode, si13, si2, **kw)
    ref = moe.moe_forward(*prob, act_quant=mode, w13_input_scale=si13, w2_input_scale=si2, b13=b13, b2=b2)
    allow = stage2_allowance(*prob, mode, si13, si2, b13=b13, h_exact=h_exact)
    if h_exact:
        # only the SiLU's rounding is left: a few single elements at most
        rms = float(np.sqrt(np.mean(ref * ref)))
        assert (allow > 0).mean() <= 0.1 and allow.max() <= 0.05 * rms
    assert_close_with_allowance(got, ref, allow)
    # not the A16W4 layer: the quantisation is applied
    plain = moe.moe_forward(*prob, b13=b13, b2=b2)
    assert moe_tolerance_report(got, plain)["n_bad"] > 0


SCHEMES = [("mxfp4", 1.0, 1.0), ("fp8", 0.125, 0.0078125)]


@pytest.mark.parametrize("mode,si13,si2", SCHEMES)
@pytest.mark.parametrize("path,T,topk", [(PATH_DECODE, 7, 4), (PATH_DECODE, 40, 4), (PATH_PREFILL, 160, 3)])
def test_layer_exact_h(mw, mode, si13, si2, path, T, topk):
    prob = exact_problem(300 + T, 8, 1024, 512, T, topk)
    check_layer(mw, prob, path, mode, si13, si2, h_exact=True)


@pytest.mark.parametrize("mode,si13,si2", SCHEMES)
def test_layer_exact_h_two_launch_decode(mw, mode, si13, si2):
    # H above 3584: gate_up and down run as two launches
    prob = exact_problem(77, 6, 4096, 512, 12, 2)
    check_layer(mw, prob, PATH_DECODE, mode, si13, si2, h_exact=True)


@pytest.mark.parametrize("mode,si13,si2", [("mxfp4", 1.0, 1.0), ("fp8", 0.02, 0.004)])
@pytest.mark.parametrize("path,T,topk", [(PATH_DECODE, 9, 4), (PATH_PREFILL, 130, 2)])
def test_layer_gaussian_with_bias(mw, mode, si13, si2, path, T, topk):
    prob = gaussian_problem(500 + T, 8, 1024, 512, T, topk)
    g = synth.rng(600 + T)
    b13 = synth.bf16_bits_from_f32(synth.gaussian(g, (8, 1024), 0.3))
    b2 = synth.bf16_bits_from_f32(synth.gaussian(g, (8, 1024), 0.3))
    check_layer(mw, prob, path, mode, si13, si2, h_exact=False, b13=b13, b2=b2)


@pytest.mark.parametrize("mode,si13,si2", SCHEMES)
def test_layer_k3_shape_sampled(mw, mode, si13, si2):
    # the 112-expert, H=3584, I=3072, top-15 layer at one token (the fused
    # decode launch), exact-h inputs, sampled outputs
    S = synth.k3(1)
    prob = exact_problem(11, S.E, S.H, S.I, S.T, S.topk)
    got = run(mw, prob, PATH_DECODE, mode, si13, si2)
    cols = np.sort(synth.rng(12).choice(S.H, 96, replace=False))
    toks = np.arange(S.T)
    ref = moe.moe_forward_sampled(*prob, toks, cols, act_quant=mode, w13_input_scale=si13, w2_input_scale=si2)
    allow = stage2_allowance(*prob, mode, si13, si2, h_exact=True, tokens=toks, cols=cols)
    assert_close_with_allowance(got[np.ix_(toks, cols)], ref, allow)


def test_act_quant_rejected_with_int4_weights(mw):
    prob = gaussian_problem(1, 4, 256, 128, 3, 2)
    x, ids, w, w13, s13, w2, s2 = prob
    q13 = torch.zeros_like(dev(w13))
    f13 = torch.ones(s13.shape, dtype=torch.float32, device="cuda")
    q2 = torch.zeros_like(dev(w2))
    f2 = torch.ones(s2.shape, dtype=torch.float32, device="cuda")
    with pytest.raises(mw.MoeError):
        mw.moe_a16w4_int4g32(bf16_dev(x), dev(ids), dev(w), q13, f13, q2, f2, act_quant="fp8")


@pytest.mark.parametrize("mode,si13,si2", [("mxfp4", 1.0, 1.0), ("fp8", 0.5, 0.004)])
@pytest.mark.parametrize("path,T,topk", [(PATH_DECODE, 7, 4), (PATH_DECODE, 40, 4), (PATH_PREFILL, 160, 3)])
def test_layer_wide_activation_range(mw, mode, si13, si2, path, T, topk):
    # every element of x scaled by its own power of two in [2^-20, 2^20]: MX
    # block scales spread over 40 binades within a row (the decode kernels'
    # f16 window), FP8 quotients from the subnormal range to saturation
    E, H, I = 8, 1024, 512
    g = synth.rng(950 + T)
    xf = synth.gaussian(g, (T, H)) * np.exp2(g.integers(-20, 21, size=(T, H))).astype(np.float32)
    x = synth.bf16_bits_from_f32(xf)
    ids, w = synth.router_topk(g, T, E, topk)
    w13, s13 = formats.quantize_mxfp4(synth.gaussian(g, (E, 2 * I, H), 0.02))
    w2, s2 = formats.quantize_mxfp4(synth.gaussian(g, (E, H, I), 0.02))
    prob = (x, ids, w, w13, s13, w2, s2)
    got = run(mw, prob, path, mode, si13, si2)
    ref = moe.moe_forward(*prob, act_quant=mode, w13_input_scale=si13, w2_input_scale=si2)
    assert np.isfinite(ref).all()
    assert_close_with_allowance(got, ref, stage2_allowance(*prob, mode, si13, si2))


@pytest.mark.parametrize("mode,si13,si2,toks", [("mxfp4", 1.0, 1.0, (0, 4095)), ("fp8", 0.125, 0.0078125, (2047,))])
def test_layer_k3_prefill_sampled(mw, mode, si13, si2, toks):
    # the tensor-core kernels at the production shape: 4096 tokens, top-15
    # with skewed routing, exact-h inputs, sampled outputs
    S = synth.k3(4096)
    g = synth.rng(21)
    x = synth.bf16_bits_from_f32(g.integers(-8, 9, size=(S.T, S.H)).astype(np.float32))
    ids, w = synth.router_topk(g, S.T, S.E, S.topk, expert_bias_std=2.0)
    w13 = g.integers(0, 256, size=(S.E, 2 * S.I, S.H // 2), dtype=np.uint8)
    w2 = g.integers(0, 256, size=(S.E, S.H, S.I // 2), dtype=np.uint8)
    s13 = g.integers(117, 122, size=(S.E, 2 * S.I, S.H // 32), dtype=np.uint8)
    s2 = g.integers(117, 122, size=(S.E, S.H, S.I // 32), dtype=np.uint8)
    prob = (x, ids, w, w13, s13, w2, s2)
    got = run(mw, prob, PATH_PREFILL, mode, si13, si2)
    toks = np.array(toks)
    cols = np.sort(synth.rng(22).choice(S.H, 64, replace=False))
    ref = moe.moe_forward_sampled(*prob, toks, cols, act_quant=mode, w13_input_scale=si13, w2_input_scale=si2)
    allow = stage2_allowance(*prob, mode, si13, si2, h_exact=True, tokens=toks, cols=cols)
    assert_close_with_allowance(got[np.ix_(toks, cols)], ref, allow)
    assert np.isfinite(got).all()
