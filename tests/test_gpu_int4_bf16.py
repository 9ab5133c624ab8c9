"""GPU parity of int4_per_group_32 with bfloat16 group scales (the "groupwise
bf16 scales" of the vLLM PR #51274 commit message) against the CPU oracle.

* requant_mxfp4_to_int4g32_bf16s bit-exact (codes and bf16 scale bits) at low,
  normal and high scale bytes, and on sampled experts of the full-size layer.
* The MoE on those weights: weight-streaming kernels (fused, routed, two
  launches), tensor-core kernels, the full-size layer sampled, and the
  checked build clean on it.
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

    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits(t):
    """bf16 tensor on the GPU -> its bit patterns (uint16) on the host."""
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def gpu_requant(mw, w, s, chunk=8):
    q, sb = mw.requant_mxfp4_to_int4g32(dev(w), dev(s), experts_per_chunk=chunk, scale_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    return q, sb


@pytest.mark.parametrize("s_lo,s_hi", [(0, 12), (100, 140), (240, 252)])
def test_requant_bf16_bitexact_scale_ranges(mw, s_lo, s_hi):
    g = synth.rng(400 + s_lo)
    w = g.integers(0, 256, size=(5, 48, 256), dtype=np.uint8)
    w[0, 0, :16] = 0  # an all-zero group
    s = g.integers(s_lo, s_hi + 1, size=(5, 48, 16), dtype=np.uint8)
    q, sb = gpu_requant(mw, w, s, chunk=2)
    rq, rs = requant.requant_mxfp4_to_int4g32(w, s, scale_dtype="bf16")
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(bits(sb), rs)


def problem(seed, E, H, I, T, topk):
    g = synth.rng(seed)
    x = synth.activations_bf16(g, T, H)
    ids, w = synth.router_topk(g, T, E, topk)
    ids[0, -1] = -1
    w13, s13 = formats.quantize_mxfp4(synth.gaussian(g, (E, 2 * I, H), 0.02))
    w2, s2 = formats.quantize_mxfp4(synth.gaussian(g, (E, H, I), 0.02))
    q13, b13 = requant.requant_mxfp4_to_int4g32(w13, s13, scale_dtype="bf16")
    q2, b2 = requant.requant_mxfp4_to_int4g32(w2, s2, scale_dtype="bf16")
    return x, ids, w, q13, b13, q2, b2


def run(mw, prob, path, workspace=None):
    x, ids, w, q13, b13, q2, b2 = prob
    bf = lambda a: dev(a.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    out = mw.moe_a16w4_int4g32(xd, dev(ids), dev(w), dev(q13), bf(b13), dev(q2), bf(b2), path=path,
                               workspace=workspace)
    torch.cuda.synchronize()
    return formats.bf16_to_f64(bits(out))


@pytest.mark.parametrize("path,E,H,I,T,topk", [
    (PATH_DECODE, 8, 512, 256, 5, 2),      # fused, in-kernel grouping
    (PATH_DECODE, 8, 1024, 512, 60, 4),    # routing kernel
    (PATH_DECODE, 4, 4096, 256, 3, 2),     # two launches
    (PATH_PREFILL, 8, 512, 512, 200, 4),   # tensor-core kernels
    (PATH_PREFILL, 5, 1024, 512, 130, 3),
])
def test_moe_int4_bf16_scales(mw, path, E, H, I, T, topk):
    prob = problem(500 + T, E, H, I, T, topk)
    assert_moe_close(run(mw, prob, path), moe.moe_forward(*prob, kind="int4g32_bf16"))


@pytest.fixture(scope="module")
def k3_bf16(mw):
    """The 112-expert, H=3584, I=3072 layer's MXFP4 bytes and their bf16-scale
    int4 requantisation on the GPU."""
    S = synth.k3(1)
    g = synth.rng(100)
    w13, s13 = synth.random_mxfp4_bytes(g, S.E, 2 * S.I, S.H)
    w2, s2 = synth.random_mxfp4_bytes(g, S.E, S.H, S.I)
    q13, b13 = gpu_requant(mw, w13, s13)
    q2, b2 = gpu_requant(mw, w2, s2)
    return (w13, s13, w2, s2), (q13, b13, q2, b2)


def _oracle_experts(host, experts):
    """The oracle's bf16-scale requantisation of the experts it needs."""
    w13, s13, w2, s2 = host
    oq13, ob13 = np.zeros_like(w13), np.zeros(s13.shape, np.uint16)
    oq2, ob2 = np.zeros_like(w2), np.zeros(s2.shape, np.uint16)
    for e in experts:
        oq13[e:e + 1], ob13[e:e + 1] = requant.requant_mxfp4_to_int4g32(w13[e:e + 1], s13[e:e + 1],
                                                                         scale_dtype="bf16")
        oq2[e:e + 1], ob2[e:e + 1] = requant.requant_mxfp4_to_int4g32(w2[e:e + 1], s2[e:e + 1], scale_dtype="bf16")
    return oq13, ob13, oq2, ob2


@pytest.mark.parametrize("T,bias,toks", [(1, None, (0,)), (1024, 2.0, (1023,))])
def test_moe_int4_bf16_scales_k3_sampled(mw, k3_bf16, T, bias, toks):
    # the full-size layer: T=1 on the fused decode launch, T=1024 with skewed
    # routing on the tensor-core kernels; the oracle requantises the experts
    # it needs from the same MXFP4 bytes
    host, (q13, b13, q2, b2) = k3_bf16
    S = synth.k3(T)
    g = synth.rng(333 + T)
    x = synth.activations_bf16(g, T, S.H)
    ids, w = synth.router_topk(g, T, S.E, S.topk, expert_bias_std=bias)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    out = mw.moe_a16w4_int4g32(xd, dev(ids), dev(w), q13, b13, q2, b2)
    torch.cuda.synchronize()
    got = formats.bf16_to_f64(bits(out))
    toks = np.array(toks)
    cols = np.sort(g.choice(S.H, 64, replace=False))
    need = sorted({int(e) for t in toks for e in ids[t]})
    oq13, ob13, oq2, ob2 = _oracle_experts(host, need)
    for e in need[:2]:  # the GPU's requantised experts are the oracle's, byte for byte
        assert np.array_equal(q13[e].cpu().numpy(), oq13[e]) and np.array_equal(bits(b13[e]), ob13[e])
    ref = moe.moe_forward_sampled(x, ids, w, oq13, ob13, oq2, ob2, toks, cols, kind="int4g32_bf16")
    assert_moe_close(got[np.ix_(toks, cols)], ref)
    assert np.isfinite(got).all()


def test_checked_build_clean_on_int4_bf16_scales(mw):
    mw.use_checked(True)
    try:
        for path, T in ((PATH_DECODE, 9), (PATH_PREFILL, 200)):
            prob = problem(700 + T, 6, 512, 512, T, 3)
            d = mw.dims(6, 512, 512, 3, T, path)
            ws = torch.zeros(mw.moe_workspace_bytes(d), dtype=torch.uint8, device="cuda")
            got = run(mw, prob, path, workspace=ws)
            assert mw.moe_read_status(d, ws) == 0
            assert_moe_close(got, moe.moe_forward(*prob, kind="int4g32_bf16"))
    finally:
        mw.use_checked(False)
