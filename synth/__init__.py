"""Seeded synthetic inputs for the A16W4 mixture-of-experts layer.

This module is shared by the tests, the smoke check and the benchmark.  It only
draws random numbers and packs them into the byte layouts the layer consumes; it
holds none of the layer's arithmetic (no E2M1/E8M0 decoding, no GEMM, no
activation, no requantisation).  The oracle quantises the Gaussian weights drawn
here into MXFP4; the benchmark, which may not call the oracle, draws MXFP4 bytes
directly with ``random_mxfp4_bytes``.

Shapes follow the MXFP4 MoE weight layout of ``Mxfp4MoEMethod.create_weights``
(vLLM quantization/mxfp4 API page): ``w13[E, 2I, H/2]`` + ``w13_scale[E, 2I, H/32]``
and ``w2[E, H, I/2]`` + ``w2_scale[E, H, I/32]``, uint8.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class MoEShape:
    """Problem size: E experts, hidden H, intermediate I, top-k, T tokens."""

    E: int
    H: int
    I: int
    topk: int
    T: int

    @property
    def P(self) -> int:
        return self.T * self.topk


# The tiny correctness case and the Kimi-K3 expert-parallel rank shape
# (112 local experts of 896, model_dim 3584, intermediate_dim 3072, top-15),
# from the production-shape validation list on the vLLM PR #51274 page.
TINY = MoEShape(E=8, H=256, I=128, topk=2, T=4)


def k3(T: int) -> MoEShape:
    return MoEShape(E=112, H=3584, I=3072, topk=15, T=T)


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def gaussian(g: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    """float32 N(0, std^2) draws."""
    return (g.standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (torch's conversion) and return the uint16 bit patterns."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def activations_bf16(g: np.random.Generator, T: int, H: int, std: float = 1.0) -> np.ndarray:
    """Token activations x ~ N(0, std^2) as bfloat16 bit patterns, uint16[T, H]."""
    return bf16_bits_from_f32(gaussian(g, (T, H), std))


def router_topk(g: np.random.Generator, T: int, E: int, topk: int,
                expert_bias_std: float | None = None):
    """Top-k routing drawn from N(0,1) router logits.

    Softmax over the E logits, keep the k largest (ties go to the lower expert
    id), renormalise the kept probabilities to sum to one.  With
    ``expert_bias_std`` a per-expert bias N(0, std^2) is added to every token's
    logits first, which makes expert loads uneven (the skewed prefill case).
    Returns ``ids int32[T, topk]`` and ``weights float32[T, topk]``.
    """
    logits = g.standard_normal(size=(T, E)).astype(np.float64)
    if expert_bias_std is not None:
        logits = logits + g.standard_normal(size=(1, E)) * expert_bias_std
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :topk]
    w = np.take_along_axis(p, order, axis=1)
    w = w / w.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


def random_mxfp4_bytes(g: np.random.Generator, E: int, N: int, K: int,
                       scale_lo: int = 116, scale_hi: int = 121):
    """MXFP4 tensors drawn directly as bytes: every nibble uniform over the 16
    codes and every E8M0 scale byte uniform in [scale_lo, scale_hi].

    Returns ``(packed uint8[E, N, K/2], scale uint8[E, N, K/32])``.
    """
    assert K % 32 == 0
    packed = g.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    scale = g.integers(scale_lo, scale_hi + 1, size=(E, N, K // 32), dtype=np.uint8)
    return packed, scale
