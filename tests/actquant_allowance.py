"""Tolerance allowance for MoE outputs whose second GEMM takes quantised
activations (W4A4 / W4A8 schemes).

The stage-1 input x is bf16, so both sides quantise it identically.  The
stage-2 input a is computed: the kernels hold it in float32 with their own
summation order, the oracle rounds its float64 value to float32.  Where a lies
so close to a rounding decision of the quantiser (an E2M1 / e4m3 midpoint, or a
power of two that moves an MX block's scale) that the kernels' float32 error
can cross it, both quantised values are correct results of the scheme.  This
module bounds the kernels' error on a, finds every element whose quantised
value is not determined by that bound, and returns, per output element, the
largest change those elements can make:

    allowance[t, m] = sum over pairs (t, k) of |w[t, k]| * sum_j |W2[e][m, j]| * range_j

with range_j the spread of the possible quantised values of a_j.  Elements
with a determined quantised value add nothing, so for most outputs the
allowance is exactly 0 and the ordinary tolerance applies.

Error bound on h = W13 x (float32 sums of exact products in any order):
16 * sqrt(K) * 2^-23 * sqrt(sum_k (x_k w_nk)^2) -- a probabilistic bound (the
rounding errors of a sum of K terms grow like sqrt(K) ulps of its partial
sums; 16 leaves many standard deviations) that also covers an accumulation
that truncates on every one of its K/16 tensor-core steps, for K <= 4096 --
plus 2^-20 |h| (scale and bias roundings), plus 2^-25 * max(1, 2^-14 *
max_k |x_k|) * sum_k |w_nk| (activations rounded to the f16 grid in the
weight-streaming kernels: unscaled, at most 2^-25 each; scaled so that the
range's largest value lies in [2^14, 2^15), at most 2^-25 of the unit that
maps to 2^-14 of it).  The worst-case bound K * 2^-23 * sum_k |x_k w_nk| would leave an
allowance on every output and test nothing.

With ``h_exact`` the caller's inputs make every product and partial sum of h
a dyadic number that float32 holds exactly (small integers times E2M1 weights
with a narrow band of scales, FP8 input scales powers of two), so h carries
no error at all, whatever the summation order, and only the SiLU's rounding
remains.  Then a = SiLU(g) u: first-order propagation, a
second-order term, and (8 + 2 min(|g|, 100)) * 2^-23 |a| for the fast
exponential and division of the kernels' SiLU (the exponential's error grows
with |g| until it underflows or overflows near |g| = 90, where SiLU(g) is g
or 0 to within an ulp).
"""

from __future__ import annotations

import numpy as np

from oracle import actquant, formats

_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e2m1_rne(r):
    """Magnitudes (float64, >= 0) -> nearest E2M1 magnitude, ties to the even
    code, saturating at 6."""
    r = np.minimum(r, 6.0)
    hi = np.clip(np.searchsorted(_E2M1_GRID, r, side="left"), 0, 7)
    lo = np.maximum(hi - 1, 0)
    d_lo = r - _E2M1_GRID[lo]
    d_hi = _E2M1_GRID[hi] - r
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    return np.where(take_hi, _E2M1_GRID[hi], _E2M1_GRID[lo])


def mx_qdq_with_scale(v, sbyte):
    """Quantise-dequantise float32-exact values v with the given E8M0 byte(s)."""
    X = np.ldexp(1.0, np.asarray(sbyte, dtype=np.int32) - 127)
    mag = _e2m1_rne(np.abs(v) / X) * X
    return np.where(np.signbit(v), -mag, mag)


def mx_scale_byte(amax):
    amax = np.asarray(amax, dtype=np.float64)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(amax > 0, amax, 1.0))).astype(np.int64) - 2
    return np.where(amax > 0, np.clip(e + 127, 0, 254), 0)


def _f32(v):
    return np.asarray(v, dtype=np.float64).astype(np.float32).astype(np.float64)


def _spread(a, da, mode, s2):
    """Per element, max - min of the quantised values reachable from [a - da, a + da]."""
    lo, hi = _f32(a - da), _f32(a + da)
    if mode == "fp8":
        return actquant.act_qdq(hi, "fp8", s2) - actquant.act_qdq(lo, "fp8", s2)
    n, I = a.shape
    blk = lambda z: z.reshape(n, I // 32, 32)  # noqa: E731
    am_lo = blk(np.maximum(np.abs(a) - da, 0.0)).max(-1)
    am_hi = blk(np.abs(a) + da).max(-1)
    sb_lo, sb_hi = mx_scale_byte(_f32(am_lo)), mx_scale_byte(_f32(am_hi))
    qmin = np.full((n, I // 32, 32), np.inf)
    qmax = np.full((n, I // 32, 32), -np.inf)
    for step in range(int((sb_hi - sb_lo).max()) + 1):
        sb = np.minimum(sb_lo + step, sb_hi)[..., None]
        qmin = np.minimum(qmin, mx_qdq_with_scale(blk(lo), sb))
        qmax = np.maximum(qmax, mx_qdq_with_scale(blk(hi), sb))
    return (qmax - qmin).reshape(n, I)


def stage2_allowance(x_bits, ids, w, w13, s13, w2, s2, mode, w13_input_scale=1.0, w2_input_scale=1.0,
                     b13=None, h_exact=False, tokens=None, cols=None):
    """float64[T, H] allowance (see the module docstring); MXFP4 weights.
    With ``tokens`` / ``cols``: only those outputs, float64[len(tokens), len(cols)]."""
    X = actquant.act_qdq(formats.bf16_to_f64(x_bits), mode, w13_input_scale)
    T, H = X.shape
    E = w13.shape[0]
    I = w13.shape[1] // 2
    ids = np.asarray(ids)
    wts = np.asarray(w, dtype=np.float32).astype(np.float64)
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    cols = np.arange(H) if cols is None else np.asarray(cols)
    X = X[tokens]
    ids = ids[tokens]
    wts = wts[tokens]
    allow = np.zeros((tokens.size, cols.size))
    for e in np.unique(ids[(ids >= 0) & (ids < E)]):
        toks, ks = np.nonzero(ids == e)
        W13 = formats.dequant_mxfp4(w13[e], s13[e])
        W2 = formats.dequant_mxfp4(w2[e][cols], s2[e][cols])
        Xe = X[toks]
        h = Xe @ W13.T
        if b13 is not None:
            h = h + formats.bf16_to_f64(b13[e])
        if h_exact:
            dh = np.zeros_like(h)
        else:
            S2 = np.sqrt((Xe * Xe) @ (W13 * W13).T)
            xmax = np.abs(Xe).max(1, keepdims=True)
            dh = (16.0 * np.sqrt(H) * 2.0 ** -23 * S2 + 2.0 ** -20 * np.abs(h)
                  + 2.0 ** -25 * np.maximum(1.0, 2.0 ** -14 * xmax) * np.abs(W13).sum(1))
        g, u, dg, du = h[:, :I], h[:, I:], dh[:, :I], dh[:, I:]
        with np.errstate(over="ignore"):  # exp(-g) = inf for very negative g: sig = 0, exactly the limit
            sig = 1.0 / (1.0 + np.exp(-g))
        silu = g * sig
        dsilu = sig * (1.0 + g * (1.0 - sig))
        a = silu * u
        da = (np.abs(dsilu) * np.abs(u) * dg + np.abs(silu) * du + dg * du + 0.5 * dg * dg * np.abs(u)
              + (8.0 + 2.0 * np.minimum(np.abs(g), 100.0)) * 2.0 ** -23 * np.abs(a))
        rng = _spread(a, da, mode, w2_input_scale)
        np.add.at(allow, toks, np.abs(wts[toks, ks])[:, None] * (rng @ np.abs(W2).T))
    return allow
