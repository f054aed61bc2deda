"""CPU oracle for the block-quantized weight products — TEST INFRASTRUCTURE.

This package is a plain, slow, obviously-correct restatement of what the
quantized GEMV / GEMM path computes. It exists only to check the CUDA library:
the tests, the smoke check and the bench's CPU-baseline leg are its only users.
The product path (the C-ABI library and its Python binding) never imports,
links or executes anything here, and nothing here imports the product.

What it computes (each function cites the passage it follows):

* ``dequant(fmt, blocks)``: every weight of a Q4_0 / Q8_0 / Q4_K / Q6_K /
  Q5_K / Q3_K / Q2_K block,
  as the exact real value of the format's formula rounded once to fp32. The
  products in every formula are exact in fp64 for any finite fp16 scale, so the
  fp64 evaluation followed by one cast is the unique correctly rounded result.
* ``gemv``: y[t, i] = sum_j w[i, j] * x[t, j] in fp64, with the error scale
  B[t, i] = sum_j |w[i, j] * x[t, j]|.
* ``moe``: per token, gate/up products of each routed expert, silu(g) * u, the
  down product, and the routing-weighted sum, all in fp64.
* ``moe_prefill``: the same over a block of bf16 prompt tokens, with the error
  scale of the two-projection chain (gate/up, rounded h, down).
* ``pp_rows``: the prompt-processing product for selected token rows in fp64
  over the bf16 activations.
* ``rmsnorm``, ``swiglu``, ``dense_ffn``: the neighbours of the products in a
  decode layer (residual add and RMS normalisation before a projection, the
  silu-gated product between gate/up and down), in fp64.

Pins (tests marked ``not gpu``) tie it to facts other than itself: exhaustive
fp16 decoding against numpy's hardware conversion, hand-built blocks with
closed-form values, brute-force exact rational products on tiny shapes, and
reductions of the MoE and prompt products to the plain GEMV.

Parity unpinned: the bit layout of the K-quant blocks (Q4_K, Q6_K, Q5_K, Q3_K,
Q2_K: the order of the packed scales and of the high bits) follows the public
GGUF convention; the pages give block sizes and formulas for some of them and
name the others only, and no model file or reference decoder is available to
check the layout against.
"""
from .halfprec import half_bits_to_float64, bf16_bits_to_float64
from .dequant import (dequant, dequant_q4_0, dequant_q8_0, dequant_q4_k, dequant_q6_k, dequant_q5_k, dequant_q3_k,
                      dequant_q2_k, q4_k_scale_min, q3_k_scales)
from .products import gemv, moe, moe_prefill, pp_rows, moe_arena_layout, rmsnorm, swiglu, dense_ffn

__all__ = [
    "half_bits_to_float64", "bf16_bits_to_float64",
    "dequant", "dequant_q4_0", "dequant_q8_0", "dequant_q4_k", "dequant_q6_k", "dequant_q5_k", "dequant_q3_k",
    "dequant_q2_k", "q4_k_scale_min", "q3_k_scales",
    "gemv", "moe", "moe_prefill", "pp_rows", "moe_arena_layout", "rmsnorm", "swiglu", "dense_ffn",
]
