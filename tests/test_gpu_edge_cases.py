"""GPU parity on the method's edge cases, against the CPU oracle.

* E8M0 scale bytes across the format's range: bytes near 0 (block scales
  2^-127.., subnormal as bf16 and as float32), bytes above 142 (the tensor-core
  converter's second multiply) and up to 250, each expert with its own band
  of scale bytes (MXFP4 scales are per 32-block, the Mxfp4MoEMethod page's
  ``create_weights``: ``w13_weight_scale`` / ``w2_weight_scale`` E8M0 per
  block of 32 along K).  Every token goes to one expert (top-1) and its
  activations are scaled by a power of two that keeps the expert's
  intermediate and output inside float32 and bf16, so each band decides its
  own tokens' outputs; the tolerance is applied band by band (RMS over that
  band's tokens), as one RMS over all tokens would be set by the largest band.
* Activations whose magnitudes span 2^-20 .. 2^20 inside every 32-element
  block and across the decode kernels' per-warp K ranges.
* The requantiser bit-exact on all 112 experts of both w13 and w2 of the
  full-size expert-parallel shape (rows sampled per expert; the oracle
  converts each sampled row).
"""

import numpy as np
import pytest
import torch

import synth
from oracle import formats, moe, requant
from tests.tolerance import assert_moe_close

pytestmark = pytest.mark.gpu

PATH_DECODE, PATH_PREFILL = 1, 2

# (w13 scale bytes, w2 scale bytes, activation exponent) per expert
BANDS = [
    ((0, 1), (200, 210), 80),      # w13 values 2^-128 .. : bf16 / float32 subnormal block scales
    ((0, 20), (150, 190), 50),     # tiny w13 scales, large w2 scales
    ((140, 175), (50, 80), 0),     # w13 above 142 (second multiply in the converter), small w2
    ((230, 250), (100, 110), -100),  # near the top of the E8M0 range, tiny activations
    ((110, 126), (110, 126), 0),   # the ordinary range, for reference
]


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


def banded_problem(seed, H, I, T):
    g = np.random.default_rng(seed)
    E = len(BANDS)
    w13 = g.integers(0, 256, size=(E, 2 * I, H // 2), dtype=np.uint8)
    w2 = g.integers(0, 256, size=(E, H, I // 2), dtype=np.uint8)
    s13 = np.zeros((E, 2 * I, H // 32), np.uint8)
    s2 = np.zeros((E, H, I // 32), np.uint8)
    for e, ((a, b), (c, d), _) in enumerate(BANDS):
        s13[e] = g.integers(a, b + 1, size=s13[e].shape)
        s2[e] = g.integers(c, d + 1, size=s2[e].shape)
    ids = g.permutation(np.arange(T) % E).astype(np.int32)[:, None]
    w = g.uniform(0.2, 1.0, size=(T, 1)).astype(np.float32)
    expo = np.array([BANDS[e][2] for e in ids[:, 0]], dtype=np.float64)
    xf = g.standard_normal((T, H)) * np.exp2(expo)[:, None]
    x = synth.bf16_bits_from_f32(xf.astype(np.float32))
    return x, ids, w, w13, s13, w2, s2


def run(mw, prob, path, kind="mxfp4"):
    x, ids, w, a, b, c, d = prob
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    fn = mw.moe_a16w4_mxfp4 if kind == "mxfp4" else mw.moe_a16w4_int4g32
    out = fn(xd, dev(ids), dev(w), dev(a), dev(b), dev(c), dev(d), path=path)
    torch.cuda.synchronize()
    return formats.bf16_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))


def assert_per_band(got, ref, ids):
    assert np.isfinite(ref).all()
    for e in range(len(BANDS)):
        rows = ids[:, 0] == e
        assert_moe_close(got[rows], ref[rows])


@pytest.mark.parametrize("path,T", [(PATH_DECODE, 60), (PATH_DECODE, 150), (PATH_PREFILL, 200)])
def test_scale_bands_mxfp4(mw, path, T):
    prob = banded_problem(31 + T, 512, 512, T)
    ref = moe.moe_forward(*prob)
    assert_per_band(run(mw, prob, path), ref, prob[1])


@pytest.mark.parametrize("path,T", [(PATH_DECODE, 60), (PATH_PREFILL, 200)])
def test_scale_bands_int4(mw, path, T):
    x, ids, w, w13, s13, w2, s2 = banded_problem(47 + T, 512, 512, T)
    q13, f13 = requant.requant_mxfp4_to_int4g32(w13, s13)
    q2, f2 = requant.requant_mxfp4_to_int4g32(w2, s2)
    prob = (x, ids, w, q13, f13, q2, f2)
    ref = moe.moe_forward(*prob, kind="int4g32")
    assert_per_band(run(mw, prob, path, kind="int4"), ref, ids)


def test_scale_bands_decode_two_launch(mw):
    # H above 3584: the gate_up and down GEMMs run as two launches
    prob = banded_problem(77, 4096, 512, 20)
    ref = moe.moe_forward(*prob)
    assert_per_band(run(mw, prob, PATH_DECODE), ref, prob[1])


@pytest.mark.parametrize("path,T,topk,lo,hi", [(PATH_DECODE, 7, 4, -20, 20), (PATH_DECODE, 40, 4, -20, 20),
                                               (PATH_PREFILL, 160, 3, -20, 20), (PATH_DECODE, 7, 4, -26, 0),
                                               (PATH_DECODE, 40, 4, -26, 0)])
def test_wide_activation_range(mw, path, T, topk, lo, hi):
    # every element of x scaled by its own power of two in [2^lo, 2^hi]; with
    # [-26, 0] each row's largest value lies in [2^-4, 2^15), where the
    # weight-streaming kernels leave activations unscaled and the smallest
    # values fall on the f16 subnormal grid
    E, H, I = 8, 1024, 512
    g = synth.rng(900 + T + lo)
    xf = synth.gaussian(g, (T, H)) * np.exp2(g.integers(lo, hi + 1, size=(T, H))).astype(np.float32)
    x = synth.bf16_bits_from_f32(xf)
    ids, w = synth.router_topk(g, T, E, topk)
    w13, s13 = formats.quantize_mxfp4(synth.gaussian(g, (E, 2 * I, H), 0.02))
    w2, s2 = formats.quantize_mxfp4(synth.gaussian(g, (E, H, I), 0.02))
    prob = (x, ids, w, w13, s13, w2, s2)
    ref = moe.moe_forward(*prob)
    assert_moe_close(run(mw, prob, path), ref)


@pytest.mark.parametrize("which", ["w13", "w2"])
def test_requant_k3_every_expert_bitexact(mw, which):
    S = synth.k3(1)
    g = synth.rng(100 if which == "w13" else 101)
    N, K = (2 * S.I, S.H) if which == "w13" else (S.H, S.I)
    w, s = synth.random_mxfp4_bytes(g, S.E, N, K)
    # scale bytes over the whole exact range, not only the benchmark's band
    s = g.integers(0, 253, size=s.shape, dtype=np.uint8)
    q, f = mw.requant_mxfp4_to_int4g32(dev(w), dev(s), experts_per_chunk=8)
    torch.cuda.synchronize()
    rows = np.stack([np.sort(g.choice(N, 64, replace=False)) for _ in range(S.E)])
    e_idx = np.arange(S.E)[:, None]
    rq, rs = requant.requant_mxfp4_to_int4g32(w[e_idx, rows], s[e_idx, rows])
    rows_t = torch.from_numpy(rows).cuda()
    e_t = torch.arange(S.E, device="cuda")[:, None]
    assert np.array_equal(q[e_t, rows_t].cpu().numpy(), rq)
    assert np.array_equal(f[e_t, rows_t].cpu().numpy().view(np.uint32), rs.view(np.uint32))
