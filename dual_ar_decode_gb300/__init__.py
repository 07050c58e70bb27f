"""GB300 (sm_103a) Dual-AR decode: thin Python binding over libtf_dualar.so.

Every step of the decode path runs in the CUDA library; this package only
marshals arguments through the C ABI declared in include/tf.h.  Importing it
does not load the library; ``binding.lib()`` does, and raises if the library
has not been built (there is no fallback).
"""
from .binding import (TF_OK, TfError, Decoder, config_from_dims, lib, library_path,
                      op_attention, op_attention_prompt, op_gemm, op_gemm_skinny, op_gemm_skinny_fp8, op_gemm_skinny_nvfp4, op_gemv, op_quantize_fp8,
                      op_quantize_nvfp4, op_select)

__all__ = ["TF_OK", "TfError", "Decoder", "config_from_dims", "lib", "library_path",
           "op_attention", "op_attention_prompt", "op_gemm", "op_gemm_skinny", "op_gemm_skinny_fp8", "op_gemm_skinny_nvfp4", "op_gemv", "op_quantize_fp8",
           "op_quantize_nvfp4", "op_select"]
