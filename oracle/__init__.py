"""CPU oracle for the Dual-AR (RQ-Transformer) decode step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it.  It shares no code with the CUDA library.

The oracle is a plain, slow restatement of what the decode step computes,
in float64 NumPy (weights are the exact bf16 / dequantised-fp8 values).
Each function cites the passage of the source pages it follows:

  * tuna-fish README (github.557886.com/reesertg/tuna-fish), sections
    "Inference estimation" (model shapes, static KV cache, bytes per step) and
    "training estimation" (slowAR tied embedding, fastAR head size);
  * "Fish Speech" tour (pyshine.com/fish-speech), "Why You Need This"
    (rotary embeddings, grouped-query attention, slow/fast heads, top-k);
  * fish-s2-pro-mlx-local-deploy README, architecture paragraph (slow AR on
    the time axis predicts the semantic codebook, fast AR the 9 residual
    codebooks; 10 codebooks at ~21 Hz);
  * drbaph s2-pro-fp8 model card, "Quantization Details" (per-row symmetric
    float8_e4m3fn weights with a float32 scale per output row).

Where the pages leave a step open, the reading taken is stated in the
docstring of the function that implements it.
"""
from .numerics import (bf16_bits_to_f64, bf16_bits_to_f32, round_to_bf16, e4m3_decode,
                       e4m3_encode_rne, fp8_quantize_rows, fp8_dequant_rows,
                       e2m1_decode, e2m1_encode_rne, nvfp4_quantize_rows, nvfp4_dequant_rows,
                       rmsnorm, rope_angles, apply_rope, attention_row,
                       causal_attention, silu, linear)
from .sampler import (philox4x32_10, exp_f32, argmax_lowest, topk_candidates,
                      topk_sample, uniform24, apply_repetition_penalty)
from .model import DualAROracle, load_formula

__all__ = [
    "bf16_bits_to_f64", "bf16_bits_to_f32", "round_to_bf16", "e4m3_decode", "e4m3_encode_rne",
    "fp8_quantize_rows", "fp8_dequant_rows", "e2m1_decode", "e2m1_encode_rne",
    "nvfp4_quantize_rows", "nvfp4_dequant_rows", "rmsnorm", "rope_angles",
    "apply_rope", "attention_row", "causal_attention", "silu", "linear", "philox4x32_10", "exp_f32",
    "argmax_lowest", "topk_candidates", "topk_sample", "uniform24",
    "apply_repetition_penalty",
    "DualAROracle", "load_formula",
]
