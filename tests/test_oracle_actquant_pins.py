"""Pins of the oracle's activation quantisers (W4A4 / W4A8 schemes) and of the
MoE with quantised activations, against library casts, closed forms and a
dense torch restatement.

* e4m3 rounding: ml_dtypes' and torch's float8_e4m3fn casts (inputs clamped to
  +-448 first: the reading saturates, the casts overflow to NaN), every finite
  code, the ties of every binade and the subnormal range.
* fp8 activation quantiser: torch float32 division and torch's cast.
* MXFP4 activation quantiser: element codes against ml_dtypes' float4_e2m1fn
  cast of v / X; the scale byte against a frexp formulation of the OCP rule
  and hand-computed cases; idempotence on the MX grid; sign of zero.
* MoE with act_quant: a dense torch path (every expert on every token, torch
  casts for the fp8 rounding) equals the oracle.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import actquant, formats, moe

E4M3_FINITE = [c for c in range(256) if c not in (0x7F, 0xFF)]


def _e4m3_values():
    return torch.tensor(E4M3_FINITE, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def _edge_floats():
    vals = _e4m3_values()
    pos = np.unique(np.abs(vals))
    mids = (pos[:-1] + pos[1:]) / 2  # every tie between neighbouring e4m3 values
    extra = np.array([448.0, 456.0, 464.0, 470.0, 480.0, 1e9, 2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -12, 1e-30, 0.0])
    base = np.concatenate([pos, mids, extra])
    return np.concatenate([base, -base, [-0.0]]).astype(np.float32)


def _random_floats(n=20000, seed=0):
    g = np.random.default_rng(seed)
    mag = np.exp2(g.uniform(-14, 10, n)) * g.uniform(1, 2, n)
    return (np.where(g.random(n) < 0.5, -1, 1) * mag).astype(np.float32)


@pytest.mark.parametrize("which", ["edges", "random"])
def test_e4m3_round_matches_ml_dtypes_and_torch(which):
    v = _edge_floats() if which == "edges" else _random_floats()
    codes, vals = actquant.e4m3_round(v.astype(np.float64))
    clamped = np.clip(v, -448, 448)
    t = torch.from_numpy(clamped).to(torch.float8_e4m3fn)
    assert np.array_equal(codes, t.view(torch.uint8).numpy())
    assert np.array_equal(vals, t.double().numpy())
    ml_dtypes = pytest.importorskip("ml_dtypes")
    assert np.array_equal(codes, clamped.astype(ml_dtypes.float8_e4m3fn).view(np.uint8))


def test_e4m3_every_finite_code_roundtrips():
    vals = _e4m3_values()
    codes, back = actquant.e4m3_round(vals)
    assert np.array_equal(codes, np.array(E4M3_FINITE, dtype=np.uint8))
    assert np.array_equal(back, vals)
    # saturation: far above the range gives +-448, code 0x7E / 0xFE
    c, q = actquant.e4m3_round(np.array([1e30, -1e30, 449.0]))
    assert list(c) == [0x7E, 0xFE, 0x7E] and list(q) == [448.0, -448.0, 448.0]


@pytest.mark.parametrize("scale", [1.0, 0.0123, 3.7e-3, 17.5])
def test_fp8_act_quant_against_torch_float32_division(scale):
    v = np.concatenate([_random_floats(4000, 3) * np.float32(scale * 50), _edge_floats() * np.float32(scale)])
    codes, deq = actquant.quantize_fp8_act(v, scale)
    r = torch.from_numpy(v) / torch.tensor(scale, dtype=torch.float32)
    t = r.clamp(-448, 448).to(torch.float8_e4m3fn)
    assert np.array_equal(codes, t.view(torch.uint8).numpy())
    assert np.array_equal(deq, t.double().numpy() * float(np.float32(scale)))


def _scale_byte_frexp(amax):
    # OCP MX shared exponent by another route: amax = m * 2^e, m in [0.5, 1),
    # so floor(log2 amax) = e - 1
    _, e = np.frexp(amax)
    return np.where(amax > 0, np.clip(e - 1 - 2 + 127, 0, 254), 0)


def test_mx_act_quant_codes_match_ml_dtypes_and_scale_rule():
    ml_dtypes = pytest.importorskip("ml_dtypes")
    g = np.random.default_rng(5)
    rows, K = 64, 256
    v = (g.standard_normal((rows, K)) * np.exp2(g.integers(-30, 30, size=(rows, K // 32)).repeat(32, 1)))
    v = v.astype(np.float32).astype(np.float64)
    v[0, :32] = 0.0            # all-zero block
    v[1, :32] = -0.0           # negative zeros
    v[2, 5] = -0.0
    v[3, :32] = 2.0 ** -140    # below the smallest scale: byte 0
    packed, sb = actquant.quantize_mxfp4_act(v)
    amax = np.abs(v).reshape(rows, K // 32, 32).max(-1)
    assert np.array_equal(sb, _scale_byte_frexp(amax).astype(np.uint8))
    X = np.ldexp(1.0, sb.astype(np.int32) - 127).repeat(32, 1)
    lib = (v / X).astype(np.float32).astype(ml_dtypes.float4_e2m1fn).view(np.uint8) & 0xF
    assert np.array_equal(formats.unpack_nibbles(packed), lib)
    assert sb[0, 0] == 0 and sb[3, 0] == 0
    assert np.all(formats.unpack_nibbles(packed)[1, :32] == 8)


def test_mx_act_scale_byte_hand_cases():
    def byte_of(amax):
        block = np.zeros(32)
        block[7] = amax
        return int(actquant.quantize_mxfp4_act(block[None])[1][0, 0])

    assert byte_of(1.0) == 125           # floor(log2 1) - 2 + 127
    assert byte_of(6.0) == 127           # largest E2M1 value at scale 1
    assert byte_of(7.99) == 127
    assert byte_of(8.0) == 128
    assert byte_of(2.0 ** -125) == 0     # -125 - 2 + 127
    assert byte_of(2.0 ** -124) == 1
    assert byte_of(3.0 * 2.0 ** 126) == 252  # 1.5 * 2^127: the largest byte a finite amax gives


def test_mx_act_quant_is_identity_on_the_grid():
    g = synth.rng(8)
    packed, sb = synth.random_mxfp4_bytes(g, 1, 16, 128)
    grid = formats.dequant_mxfp4(packed[0], sb[0])
    back = actquant.act_qdq(grid, actquant.ACT_MXFP4)
    assert np.array_equal(back, grid)


def _torch_qdq(v, mode, scale):
    """Quantise-dequantise through torch / ml_dtypes casts."""
    if mode == "fp8":
        r = torch.from_numpy(np.asarray(v, np.float32)) / torch.tensor(scale, dtype=torch.float32)
        return r.clamp(-448, 448).to(torch.float8_e4m3fn).double().numpy() * float(np.float32(scale))
    ml_dtypes = pytest.importorskip("ml_dtypes")
    v = np.asarray(v, np.float64)
    blocks = v.reshape(v.shape[:-1] + (-1, 32))
    sb = _scale_byte_frexp(np.abs(blocks).max(-1))
    X = np.ldexp(1.0, sb.astype(np.int32) - 127)[..., None]
    q = (blocks / X).astype(np.float32).astype(ml_dtypes.float4_e2m1fn).astype(np.float64)
    return (q * X).reshape(v.shape)


def _dense_torch_act_quant(x, ids, w, w13, s13, w2, s2, mode, si13, si2):
    X = torch.from_numpy(_torch_qdq(formats.bf16_to_f64(x), mode, si13))
    W13 = torch.from_numpy(formats.dequant_mxfp4(w13, s13))
    W2 = torch.from_numpy(formats.dequant_mxfp4(w2, s2))
    E, I = W13.shape[0], W13.shape[1] // 2
    out = torch.zeros(X.shape, dtype=torch.float64)
    for e in range(E):
        h = torch.nn.functional.linear(X, W13[e])
        a = torch.nn.functional.silu(h[:, :I]) * h[:, I:]
        aq = torch.from_numpy(_torch_qdq(a.numpy().astype(np.float32), mode, si2))
        y = torch.nn.functional.linear(aq, W2[e])
        for t in range(ids.shape[0]):
            for k in range(ids.shape[1]):
                if ids[t, k] == e:
                    out[t] += float(w[t, k]) * y[t]
    return out.numpy()


@pytest.mark.parametrize("mode,si13,si2", [("fp8", 0.02, 0.004), ("fp8", 1.0, 1.0), ("mxfp4", 1.0, 1.0)])
def test_moe_act_quant_matches_dense_torch(mode, si13, si2):
    g = synth.rng(31)
    E, H, I, T, topk = 6, 128, 64, 7, 2
    x = synth.activations_bf16(g, T, H)
    ids, w = synth.router_topk(g, T, E, topk)
    ids[2, 1] = -1
    w13, s13 = formats.quantize_mxfp4(synth.gaussian(g, (E, 2 * I, H), 0.05))
    w2, s2 = formats.quantize_mxfp4(synth.gaussian(g, (E, H, I), 0.05))
    ours = moe.moe_forward(x, ids, w, w13, s13, w2, s2, act_quant=mode, w13_input_scale=si13, w2_input_scale=si2)
    ref = _dense_torch_act_quant(x, ids, w, w13, s13, w2, s2, mode, si13, si2)
    assert np.allclose(ours, ref, rtol=1e-12, atol=1e-14)
    # the quantisation changes the result (the test is not vacuous)
    plain = moe.moe_forward(x, ids, w, w13, s13, w2, s2)
    assert not np.allclose(ours, plain, rtol=1e-4, atol=0)


def test_moe_act_quant_sampled_matches_full():
    g = synth.rng(41)
    E, H, I, T, topk = 5, 96, 64, 6, 3
    x = synth.activations_bf16(g, T, H)
    ids, w = synth.router_topk(g, T, E, topk)
    w13, s13 = formats.quantize_mxfp4(synth.gaussian(g, (E, 2 * I, H), 0.05))
    w2, s2 = formats.quantize_mxfp4(synth.gaussian(g, (E, H, I), 0.05))
    for mode, a, b in [("fp8", 0.01, 0.003), ("mxfp4", 1.0, 1.0)]:
        full = moe.moe_forward(x, ids, w, w13, s13, w2, s2, act_quant=mode, w13_input_scale=a, w2_input_scale=b)
        toks, cols = np.array([0, 3, 5]), np.array([1, 17, 40, 95])
        part = moe.moe_forward_sampled(x, ids, w, w13, s13, w2, s2, toks, cols, act_quant=mode,
                                       w13_input_scale=a, w2_input_scale=b)
        assert np.allclose(part, full[np.ix_(toks, cols)], rtol=1e-12, atol=1e-15)


def test_moe_act_quant_rejects_router_weight_on_input():
    g = synth.rng(2)
    x = synth.activations_bf16(g, 2, 64)
    ids, w = synth.router_topk(g, 2, 2, 1)
    w13, s13 = formats.quantize_mxfp4(synth.gaussian(g, (2, 64, 64), 0.05))
    w2, s2 = formats.quantize_mxfp4(synth.gaussian(g, (2, 64, 32), 0.05))
    with pytest.raises(ValueError):
        moe.moe_forward(x, ids, w, w13, s13, w2, s2, router_weight_on_input=True, act_quant="fp8")
