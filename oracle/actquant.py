"""Activation quantisation of the W4A4 / W4A8 schemes (oracle; test infrastructure only).

Source: vLLM PR #39136 ("[ROCm][Quantization][2/N] Refactor quark_moe w4a8 w/
oracle"), Summary and review: the OCP MX schemes ``w_mxfp4_a_mxfp4`` (MXFP4
weights and MXFP4 activations, W4A4) and ``w_mxfp4_a_fp8`` (MXFP4 weights with
*static* FP8 activations, W4A8, which needs the layer's input scales).  The
pages give the scheme names only; the readings used here:

* MXFP4 activations: every run of 32 consecutive values along the reduction
  dimension of a row shares one E8M0 scale, chosen by the OCP MX v1.0 rule
  (the same rule ``formats.quantize_mxfp4`` applies to weights): scale byte
  floor(log2(amax)) - 2 + 127 clamped to [0, 254] (byte 0 for an all-zero
  block); each value divided by the scale is rounded to the nearest E2M1 value,
  ties to the even code, saturating at 6.  The code keeps the sign bit of its
  input (-0.0 encodes as the negative zero code 8).
* FP8 activations: one static float32 scale ``s`` per GEMM input (the
  ``w13`` input and the ``w2`` input).  r = fl32(v / s) (float32 division,
  correctly rounded), then r rounded to the nearest float8 e4m3fn value, ties
  to even, saturating at +-448 (the format's largest finite value); the
  dequantised value is that e4m3 value times ``s``.
* Where the value being quantised is computed (the SiLU-gated intermediate),
  the quantiser takes it in float32: the oracle rounds its float64
  intermediate to float32 first, the precision the kernels compute it in.

Pinned by tests/test_oracle_actquant_pins.py against ml_dtypes / torch casts, closed
forms of the scale rule and every finite e4m3 code.
"""

from __future__ import annotations

import numpy as np

from . import formats

ACT_NONE, ACT_MXFP4, ACT_FP8 = "bf16", "mxfp4", "fp8"

E4M3_MAX = 448.0
_E4M3_MIN_NORMAL_EXP = -6  # smallest normal 2^-6; subnormal quantum 2^-9


def quantize_mxfp4_act(v: np.ndarray):
    """Rows of activations [..., K] -> (packed E2M1 uint8[..., K/2], E8M0
    uint8[..., K/32]).  The OCP MX rule of ``formats.quantize_mxfp4``, with the
    sign bit of every code taken from its input (so -0.0 gives code 8)."""
    v = np.asarray(v, dtype=np.float64)
    packed, sbytes = formats.quantize_mxfp4(v)
    codes = formats.unpack_nibbles(packed)
    codes = np.where(np.signbit(v), codes | 8, codes).astype(np.uint8)
    return formats.pack_nibbles(codes), sbytes


def e4m3_round(r: np.ndarray):
    """float values (float32-representable) -> (e4m3fn codes uint8, values
    float64): round to nearest even at the e4m3 quantum of the value's binade
    (2^(e-3) for |r| in [2^e, 2^(e+1)), e >= -6; 2^-9 below 2^-6), saturating
    at +-448.  The sign bit follows the input."""
    r = np.asarray(r, dtype=np.float64)
    a = np.minimum(np.abs(r), E4M3_MAX)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0))).astype(np.int64)
    e = np.maximum(e, _E4M3_MIN_NORMAL_EXP)
    quantum = np.ldexp(1.0, (e - 3).astype(np.int32))
    mag = np.round(a / quantum) * quantum  # np.round: half to even
    # codes from the rounded magnitude (it may have moved up one binade)
    normal = mag >= 2.0 ** _E4M3_MIN_NORMAL_EXP
    with np.errstate(divide="ignore"):
        ef = np.where(normal, np.floor(np.log2(np.where(normal, mag, 1.0))).astype(np.int64) + 7, 0)
    mant = np.where(normal, mag / np.ldexp(1.0, (ef - 10).astype(np.int32)) - 8, mag / 2.0 ** -9)
    codes = (np.where(np.signbit(r), 0x80, 0) | (ef << 3) | mant.astype(np.int64)).astype(np.uint8)
    return codes, np.where(np.signbit(r), -mag, mag)


def quantize_fp8_act(v: np.ndarray, scale: float):
    """Activations (float32-representable) -> (e4m3fn codes, dequantised
    float64 values q * scale), with r = fl32(v / scale)."""
    s = np.float32(scale)
    with np.errstate(over="ignore"):  # a quotient beyond float32 is inf, and saturates
        r = np.asarray(v, dtype=np.float32) / s  # IEEE float32 division
    codes, q = e4m3_round(r.astype(np.float64))
    return codes, q * np.float64(s)


def act_qdq(v: np.ndarray, mode: str, scale: float = 1.0) -> np.ndarray:
    """Quantise-dequantise rows [..., K] of activations: the values the GEMM
    multiplies under each scheme (float64).  ``v`` must be float32-exact."""
    if mode == ACT_NONE or mode is None:
        return np.asarray(v, dtype=np.float64)
    if mode == ACT_MXFP4:
        packed, sb = quantize_mxfp4_act(v)
        return formats.dequant_mxfp4(packed, sb)
    if mode == ACT_FP8:
        return quantize_fp8_act(v, scale)[1]
    raise ValueError(mode)
