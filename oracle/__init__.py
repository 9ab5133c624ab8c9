"""CPU oracle for the A16W4 MXFP4 mixture-of-experts layer (TEST INFRASTRUCTURE).

This package is a plain, slow, obviously-correct restatement of what the GPU
library computes.  It exists only to check that library: it is imported by
``tests/``, by ``__graft_entry__.smoke()`` and by the CPU-baseline leg of
``bench.py`` — never by the library itself, which has no CPU fallback.  It
shares no code with the CUDA path (no kernels, headers, tables or helpers).

Sources, all on the pages the library follows:

* vLLM ``Mxfp4MoEMethod`` API page (quantization/mxfp4):
  ``create_weights`` fixes the byte layouts (uint8 ``w13[E, 2I, H/2]``,
  ``w13_weight_scale[E, 2I, H/32]``, ``w2[E, H, I/2]``, ``w2_weight_scale[E, H, I/32]``,
  ``mxfp4_block = 32``); ``_setup_kernel_k3_situ_gfx942`` gives the requantisation
  steps (``mxfp4_to_f32`` -> ``e8m0_to_f32`` -> per-32 multiply -> bfloat16 ->
  ``per_1x32_i4_quant``, eight experts per chunk); ``apply`` gives the forward
  call (``topk_weights``, ``topk_ids``, gate_up ``w13``, down ``w2``);
  ``get_fused_moe_quant_config`` names the W4A16 emulation semantics (weights
  dequantised, activations kept in BF16).
* vLLM PR #51274 page: the stage-1 GEMM with a SiLU-gated activation, the
  production expert-parallel shape, the lossy opt-in int4_per_group_32 path.

Modules:
  formats  - E2M1 / E8M0 / bf16 decoding, MXFP4 dequantisation and quantisation
  route    - stable token->expert grouping
  moe      - the fused MoE forward (MXFP4 and int4 weights), full and sampled
  requant  - MXFP4 -> int4_per_group_32 requantisation

Numerics: the MoE is computed in float64 (x is exact bfloat16, weights are
exact after decoding); the requantiser works in float32 because the rule it
follows (scale = amax / 7, q = round-half-even(w / scale)) fixes float32.
"""

from . import formats, route, moe, requant  # noqa: F401
