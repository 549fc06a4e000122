"""GB300 (sm_103a) W8A8 INT8 linear layer.

Per-token activation quantization and a fused int8 x int8 -> int32 GEMM whose
epilogue applies the per-token x per-channel dequantization and the bias and
writes bf16 ("Realizing Native INT8 Compute for Diffusion Transformers on
Consumer GPUs: A Fused INT8 GEMM Kernel for Ideogram 4.0", arXiv 2606.14598,
abstract).  The computation lives in libi8.so (CUDA, include/i8.h); the
functions below are its torch-tensor binding.
"""
from .binding import (I8Error, e4m3_workspace_bytes, f16codes_workspace_bytes,
                      gelu_quant_act_pertoken, gemm_dequant_bias_bf16_f16codes,
                      gemm_int32_f16codes, get_option, linear_f16codes,
                      quant_act_pertoken_f16codes, gemm_dequant_bias_bf16,
                      gemm_e4m3_dequant_bias_bf16, gemm_e4m3_f32, gemm_int32,
                      layernorm_quant_act_pertoken, linear, linear_e4m3, load, plan_query,
                      quant_act_pertoken,
                      quant_act_pertoken_e4m3, quant_weight_perchannel,
                      quant_weight_perchannel_e4m3, set_option, sync_check, widen_weight_codes,
                      workspace_bytes)

__all__ = [
    "I8Error", "e4m3_workspace_bytes", "f16codes_workspace_bytes", "gelu_quant_act_pertoken",
    "gemm_dequant_bias_bf16_f16codes", "gemm_int32_f16codes", "get_option", "linear_f16codes",
    "quant_act_pertoken_f16codes", "gemm_dequant_bias_bf16", "gemm_e4m3_dequant_bias_bf16",
    "gemm_e4m3_f32", "gemm_int32", "layernorm_quant_act_pertoken", "linear", "linear_e4m3", "load", "plan_query", "quant_act_pertoken",
    "quant_act_pertoken_e4m3", "quant_weight_perchannel", "quant_weight_perchannel_e4m3",
    "set_option", "sync_check", "widen_weight_codes", "workspace_bytes",
]
