"""Element and scale formats of MXFP4 weights (oracle; test infrastructure only).

MXFP4 as used by ``Mxfp4MoEMethod`` (vLLM quantization/mxfp4 API page): packed
E2M1 elements viewed as ``torch.float4_e2m1fn_x2`` (two per uint8 byte), one
E8M0 scale viewed as ``torch.float8_e8m0fnu`` per block of ``mxfp4_block = 32``
elements along K.  ``_setup_kernel_k3_situ_gfx942`` decodes them with
``mxfp4_to_f32`` and ``e8m0_to_f32`` and multiplies each 32-block of elements by
its scale.  The pages print neither value table; the readings used here are
the OCP Microscaling (MX) v1.0 definitions those dtypes implement:

* E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit, no inf/NaN.
  Exponent field 0 is subnormal: value = mantissa * 0.5.
* E8M0: unsigned 8-bit exponent, value 2**(e - 127); e = 255 is NaN.
* Packing: element 2j is the low nibble of byte j, element 2j+1 the high nibble.
"""

from __future__ import annotations

import numpy as np

MX_BLOCK = 32  # ``mxfp4_block = 32`` in Mxfp4MoEMethod.create_weights


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    """Value of each 4-bit E2M1 code (0..15) as float64, from the field definition."""
    c = np.asarray(codes).astype(np.int64)
    sign = np.where((c >> 3) & 1, -1.0, 1.0)
    exp = (c >> 1) & 3
    man = (c & 1).astype(np.float64)
    mag = np.where(exp == 0, man * 0.5, np.ldexp(1.0 + man / 2.0, (exp - 1).astype(np.int32)))
    return sign * mag


def e8m0_decode(scale_bytes: np.ndarray) -> np.ndarray:
    """2**(e - 127) as float64 for each E8M0 byte; 255 decodes to NaN."""
    e = np.asarray(scale_bytes).astype(np.int64)
    v = np.ldexp(1.0, (e - 127).astype(np.int32))
    return np.where(e == 255, np.nan, v)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    """uint8[..., K/2] -> codes uint8[..., K]; low nibble first."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0x0F
    out[..., 1::2] = p >> 4
    return out


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """codes uint8[..., K] (each < 16) -> uint8[..., K/2]; element 2j in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    assert c.shape[-1] % 2 == 0
    return (c[..., 0::2] & 0x0F) | ((c[..., 1::2] & 0x0F) << 4)


def dequant_mxfp4(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dequantise MXFP4 rows: uint8[..., N, K/2] + uint8[..., N, K/32] -> float64[..., N, K].

    Each 32-element block along K is multiplied by its E8M0 scale, the
    ``weight_f32.view(..., K // 32, 32) * scale_f32.view(..., K // 32, 1)`` step of
    ``_setup_kernel_k3_situ_gfx942``.
    """
    vals = e2m1_decode(unpack_nibbles(packed))
    K = vals.shape[-1]
    assert scales.shape[-1] * MX_BLOCK == K, (scales.shape, K)
    blocks = vals.reshape(vals.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    sc = e8m0_decode(scales)[..., None]
    return (blocks * sc).reshape(vals.shape)


# E2M1 magnitudes in code order 0..7 (code = exponent<<1 | mantissa).
_E2M1_MAG = e2m1_decode(np.arange(8))


def quantize_mxfp4(w: np.ndarray):
    """Quantise float weights [..., N, K] to MXFP4 (input synthesis for the tests).

    OCP MX v1.0 conversion: for each 32-block the shared scale is
    X = 2**(floor(log2(amax)) - 2) (2 = E2M1's largest exponent), stored as the
    E8M0 byte floor(log2(amax)) - 2 + 127 clamped to [0, 254]; each element v/X
    is rounded to the nearest E2M1 value, ties to the even code (mantissa 0),
    and magnitudes above 6 saturate to 6.  An all-zero block gets scale byte 0.
    Returns ``(packed uint8[..., N, K/2], scales uint8[..., N, K/32])``.
    """
    w = np.asarray(w, dtype=np.float64)
    K = w.shape[-1]
    assert K % MX_BLOCK == 0
    blocks = w.reshape(w.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    amax = np.abs(blocks).max(axis=-1)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(amax > 0, amax, 1.0))).astype(np.int64) - 2
    sbyte = np.where(amax > 0, np.clip(e + 127, 0, 254), 0).astype(np.uint8)
    X = np.ldexp(1.0, sbyte.astype(np.int32) - 127)[..., None]
    r = np.abs(blocks) / X
    lo = np.clip(np.searchsorted(_E2M1_MAG, r, side="right") - 1, 0, 7)
    hi = np.minimum(lo + 1, 7)
    d_lo = r - _E2M1_MAG[lo]
    d_hi = _E2M1_MAG[hi] - r
    take_hi = (hi != lo) & ((d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0)))
    mag = np.where(take_hi, hi, lo)
    codes = (mag | np.where(blocks < 0, 8, 0)).astype(np.uint8)
    codes = codes.reshape(w.shape)
    return pack_nibbles(codes), sbyte


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64, exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f32_to_bf16_rne(a: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bits, round to nearest even (finite inputs)."""
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)
