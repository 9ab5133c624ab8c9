"""Fused A16W4 mixture-of-experts forward (oracle; test infrastructure only).

What is computed, per the pages:

* ``Mxfp4MoEMethod.apply`` (vLLM quantization/mxfp4 API page) runs the fused
  MoE on ``x`` with ``w1 = w13`` (fused gate_up projection, ``create_weights``:
  rows [0, I) gate, rows [I, 2I) up) and ``w2`` (down projection), given
  ``topk_ids`` and ``topk_weights``; ``apply_router_weight_on_input`` is off, so
  the router weight scales each expert's output.
* The W4A16 emulation backend (``get_fused_moe_quant_config``) keeps the BF16
  activations and dequantises only the weights: that is the semantics here.
* The stage-1 activation is SiLU-gated (PR #51274 page: the packed-int4 stage1
  computes SiLU; SiTUv2's formula is not on the pages, so it is not modelled):
  a = SiLU(gate) * up with SiLU(z) = z / (1 + exp(-z)).

For each pair (t, k) with e = topk_ids[t, k] in [0, E):
    h = W13[e] @ x[t]                (2I values)
    a = SiLU(h[:I]) * h[I:]
    y = W2[e] @ a                    (H values)
    out[t] += topk_weights[t, k] * y  (k ascending)
All in float64 from exact inputs.  Pairs with invalid ids add nothing.

Optional variants (not on the benchmarked path):
* biases: ``create_weights`` registers ``w13_bias`` bf16[E, 2I] and
  ``w2_bias`` bf16[E, H] when the layer has biases, and
  ``get_fused_moe_quant_config`` hands them to the kernel as ``w1_bias`` /
  ``w2_bias``.  The pages print no formula; read as the bias of each linear
  map: h = W13[e] @ x[t] + b13[e], y = W2[e] @ a + b2[e].
* ``apply_router_weight_on_input`` (``apply``): read as x[t] scaled by the
  pair's router weight before stage 1, and the combine summing the pairs'
  outputs unweighted.
* ``expert_map`` (``apply``, expert parallelism): global ids mapped to local
  ids (or -1) before the grouping, as in ``route.route``.
* ``swiglu_limit`` (``Mxfp4MoEMethod.get_fused_moe_quant_config`` passes the
  layer's ``swiglu_limit`` on as ``gemm1_clamp_limit``; no formula is
  printed): read as the gate_up GEMM's output, bias included, clamped to
  [-limit, limit] element by element before the SiLU gating.
* ``act_quant`` (vLLM PR #39136, the ``w_mxfp4_a_mxfp4`` and ``w_mxfp4_a_fp8``
  schemes): both GEMMs take quantised-dequantised activations,
  ``actquant.act_qdq``; the stage-1 input is x (bf16, exact in float32), the
  stage-2 input the intermediate a rounded to float32; W4A8 uses the static
  input scales ``w13_input_scale`` / ``w2_input_scale``.
"""

from __future__ import annotations

import numpy as np

from . import actquant, formats
from .route import local_ids, route


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def _expert_mlp(X: np.ndarray, W13: np.ndarray, W2: np.ndarray, b13=None, b2=None,
                act_quant=None, s13: float = 1.0, s2: float = 1.0, limit=None) -> np.ndarray:
    I = W13.shape[0] // 2
    if act_quant:
        X = actquant.act_qdq(X, act_quant, s13)
    h = X @ W13.T
    if b13 is not None:
        h = h + b13
    if limit is not None:
        h = np.clip(h, -limit, limit)
    a = silu(h[:, :I]) * h[:, I:]
    if act_quant:
        a = actquant.act_qdq(a.astype(np.float32), act_quant, s2)
    y = a @ W2.T
    if b2 is not None:
        y = y + b2
    return y


def _bias_rows(b_bits, e):
    return None if b_bits is None else formats.bf16_to_f64(np.asarray(b_bits)[e])


def dequant_int4(q_packed: np.ndarray, scales_f32: np.ndarray) -> np.ndarray:
    """int4_per_group_32 weights -> float64: two's-complement nibble (element 2j
    low) times the float32 scale of its 32-group."""
    codes = formats.unpack_nibbles(q_packed).astype(np.int64)
    vals = np.where(codes >= 8, codes - 16, codes).astype(np.float64)
    K = vals.shape[-1]
    blocks = vals.reshape(vals.shape[:-1] + (K // formats.MX_BLOCK, formats.MX_BLOCK))
    return (blocks * np.asarray(scales_f32, dtype=np.float32).astype(np.float64)[..., None]).reshape(vals.shape)


def _deq(kind: str, w: np.ndarray, s: np.ndarray) -> np.ndarray:
    if kind == "mxfp4":
        return formats.dequant_mxfp4(w, s)
    if kind == "int4g32":
        return dequant_int4(w, s)
    if kind == "int4g32_bf16":  # scales as bfloat16 bit patterns
        return dequant_int4(w, formats.bf16_to_f64(s).astype(np.float32))
    raise ValueError(kind)


def moe_forward(x_bits, topk_ids, topk_w, w13, s13, w2, s2, kind: str = "mxfp4", b13=None, b2=None,
                router_weight_on_input: bool = False, expert_map=None, act_quant=None,
                w13_input_scale: float = 1.0, w2_input_scale: float = 1.0, swiglu_limit=None) -> np.ndarray:
    """Full MoE output, float64[T, H].  ``x_bits`` are bfloat16 bit patterns
    uint16[T, H]; ``b13`` / ``b2`` optional bias bit patterns uint16[E, 2I] /
    uint16[E, H]; ``expert_map`` optional int32[global experts] (global id ->
    local id or -1); ``act_quant`` None, "mxfp4" or "fp8" (static scales
    ``w13_input_scale``, ``w2_input_scale``)."""
    if act_quant and router_weight_on_input:
        raise ValueError("router weight on the input with quantised activations is not modelled")
    X = formats.bf16_to_f64(x_bits)
    T, H = X.shape
    ids = np.asarray(topk_ids)
    topk = ids.shape[1]
    E = w13.shape[0]
    w = np.asarray(topk_w, dtype=np.float32).astype(np.float64)
    counts, offsets, sorted_pair, _ = route(ids, E, expert_map)
    y = np.zeros((T * topk, H), dtype=np.float64)
    for e in range(E):
        pairs = sorted_pair[offsets[e]:offsets[e + 1]]
        if pairs.size == 0:
            continue
        W13 = _deq(kind, w13[e], s13[e])
        W2 = _deq(kind, w2[e], s2[e])
        Xp = X[pairs // topk]
        if router_weight_on_input:
            Xp = Xp * w.reshape(-1)[pairs][:, None]
        y[pairs] = _expert_mlp(Xp, W13, W2, _bias_rows(b13, e), _bias_rows(b2, e), act_quant,
                               w13_input_scale, w2_input_scale, swiglu_limit)
    out = np.zeros((T, H), dtype=np.float64)
    for k in range(topk):
        out += y[k::topk] if router_weight_on_input else w[:, k:k + 1] * y[k::topk]
    return out


def moe_forward_sampled(x_bits, topk_ids, topk_w, w13, s13, w2, s2, tokens, cols,
                        kind: str = "mxfp4", expert_map=None, act_quant=None,
                        w13_input_scale: float = 1.0, w2_input_scale: float = 1.0) -> np.ndarray:
    """out[tokens][:, cols] only, float64[len(tokens), len(cols)].

    Each selected token's pairs need their full stage-1 output, but only the
    selected rows of W2; used to check full-size problems element by element.
    """
    X = formats.bf16_to_f64(x_bits)
    if act_quant:
        X = actquant.act_qdq(X, act_quant, w13_input_scale)
    ids = local_ids(topk_ids, expert_map)
    topk = ids.shape[1]
    E = w13.shape[0]
    I = w13.shape[1] // 2
    w = np.asarray(topk_w, dtype=np.float32).astype(np.float64)
    tokens = np.asarray(tokens)
    cols = np.asarray(cols)
    out = np.zeros((tokens.size, cols.size), dtype=np.float64)
    need = sorted({int(e) for t in tokens for e in ids[t] if 0 <= e < E})
    for e in need:
        W13 = _deq(kind, w13[e], s13[e])
        W2c = _deq(kind, w2[e][cols], s2[e][cols])
        for i, t in enumerate(tokens):
            for k in range(topk):
                if ids[t, k] != e:
                    continue
                h = W13 @ X[t]
                a = silu(h[:I]) * h[I:]
                if act_quant:
                    a = actquant.act_qdq(a.astype(np.float32), act_quant, w2_input_scale)
                out[i] += w[t, k] * (W2c @ a)
    return out
