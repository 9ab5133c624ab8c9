"""MXFP4 -> int4_per_group_32 requantisation (oracle; test infrastructure only).

Steps, in the order of ``Mxfp4MoEMethod._setup_kernel_k3_situ_gfx942`` (vLLM
quantization/mxfp4 API page) and the "convert eight experts at a time" change
of PR #51274:

1. for each chunk of ``experts_per_chunk`` experts (8 on the pages):
2.   decode the E2M1 elements to float32 (``mxfp4_to_f32``) and the E8M0
     scales (``e8m0_to_f32``), multiply each 32-block by its scale;
3.   cast to bfloat16 (``.to(torch.bfloat16)``);
4.   quantise every 32-group along K (``per_1x32_i4_quant``).

Step 4's rounding rule is not printed on the pages.  Reading used (symmetric
int4, float32 scale):  amax = max |w| over the group;  scale = fl32(amax / 7)
(IEEE float32 division, round to nearest even);  q = rint(w / scale) with IEEE
float32 division and round-half-to-even, clamped to [-8, 7];  an all-zero group
gets scale 0 and q = 0.

bf16 scales (the PR #51274 commit message converts to int4 "with groupwise
bf16 scales"; the benchmarked reading stores float32): the group scale is
stored as bf16, rounded to nearest even from fl32(amax / 7), and the elements
are quantised against that stored scale, q = rint(fl32(w / scale_bf16)),
so that dequantisation q * scale uses the scale the quantiser used.

Output layout (canonical, unshuffled): ``q uint8[E, N, K/2]`` with the
two's-complement code of element 2j in the low nibble, and ``scale
float32[E, N, K/32]``.  The AITER shuffles on the page are a kernel-specific
re-layout and are not modelled.

Element values E2M1 * 2**(s - 127) carry at most two significant bits and lie
in float32's exponent range, which bfloat16 shares, so step 3 leaves them
unchanged; the cast is still performed here as a separate step.
"""

from __future__ import annotations

import numpy as np

from . import formats


def _to_bf16_f32(a: np.ndarray) -> np.ndarray:
    bits = formats.f32_to_bf16_rne(a)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def quantize_int4_group32(w_f32: np.ndarray, scale_dtype: str = "f32"):
    """Symmetric int4 per 32-group along the last axis, float32 arithmetic.
    ``scale_dtype`` "bf16": the scale is rounded to bfloat16 (nearest even)
    before the elements are divided by it."""
    w = np.asarray(w_f32, dtype=np.float32)
    K = w.shape[-1]
    g = w.reshape(w.shape[:-1] + (K // 32, 32))
    amax = np.abs(g).max(axis=-1)
    scale = (amax / np.float32(7.0)).astype(np.float32)
    if scale_dtype == "bf16":
        scale = _to_bf16_f32(scale)
    elif scale_dtype != "f32":
        raise ValueError(scale_dtype)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    with np.errstate(invalid="ignore"):
        ratio = (g / safe[..., None]).astype(np.float32)
    q = np.clip(np.rint(ratio), -8, 7).astype(np.int64)
    q = np.where(scale[..., None] > 0, q, 0)
    return q.reshape(w.shape), scale


def pack_int4(q: np.ndarray) -> np.ndarray:
    """Signed int4 values [-8, 7] -> two's-complement nibbles, element 2j low."""
    return formats.pack_nibbles((np.asarray(q, dtype=np.int64) & 0xF).astype(np.uint8))


def requant_mxfp4_to_int4g32(w: np.ndarray, scale: np.ndarray, experts_per_chunk: int = 8,
                             scale_dtype: str = "f32"):
    """MXFP4 ``w uint8[E, N, K/2]`` + ``scale uint8[E, N, K/32]`` ->
    ``(q uint8[E, N, K/2], s float32[E, N, K/32])``; with ``scale_dtype``
    "bf16" the scales come back as bfloat16 bit patterns uint16[E, N, K/32]."""
    E, N, Kh = w.shape
    K = Kh * 2
    out_q = np.empty((E, N, Kh), dtype=np.uint8)
    out_s = np.empty((E, N, K // 32), dtype=np.float32)
    for lo in range(0, E, experts_per_chunk):
        hi = min(lo + experts_per_chunk, E)
        vals = formats.e2m1_decode(formats.unpack_nibbles(w[lo:hi])).astype(np.float32)
        sc = formats.e8m0_decode(scale[lo:hi]).astype(np.float32)
        blocks = vals.reshape(hi - lo, N, K // 32, 32) * sc[..., None]
        w_bf16 = _to_bf16_f32(blocks.reshape(hi - lo, N, K))
        q, s = quantize_int4_group32(w_bf16, scale_dtype)
        out_q[lo:hi] = pack_int4(q)
        out_s[lo:hi] = s
    if scale_dtype == "bf16":  # exact: the scales are bfloat16 values
        return out_q, (out_s.view(np.uint32) >> 16).astype(np.uint16)
    return out_q, out_s
