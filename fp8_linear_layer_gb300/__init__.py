"""GB300 (sm_103a) block-scaled FP8 GEMMs for a training linear layer.

Y = X W^T + b: the forward GEMM with bias / tanh-GELU epilogues, the data-
gradient GEMM with the GELU-derivative and bias-gradient epilogue, and the
accumulating fp32 weight-gradient GEMM plus its k-grouped MoE variant (and the
same GEMMs on MXFP8 operands, scaled by the tensor core), all in
hand-written CUDA behind the C ABI of include/fp8ll.h.  This package is the
Python binding (ctypes) over that library (``binding``) and the training
step of one layer built from those calls (``linear``).
"""
from .binding import (ACC_FAST, ACC_FULL, E4M3, E5M2, EPI_BIAS, EPI_BIAS_GELU, EPI_DGELU, EPI_DGELU_BGRAD,
                      EPI_NONE, EXPORTS, Fp8Error, Fp8Tensor, cast_f32, debug_starve_next_gemm, device_status,
                      empty_fp8, gemm_dgrad, gemm_dgrad_quant, gemm_fprop, gemm_wgrad, grouped_wgrad, lib, quantize, quantize_dual,
                      scale_ld, status_string, workspace_size, Fp8MxTensor, empty_mx, mx_gemm_dgrad, mx_gemm_fprop,
                      mx_gemm_wgrad, mx_quantize, mx_sf_bytes, Fp8TensorScaled, amax_history_update,
                      empty_tensor_scaled, tensor_amax, tensor_gemm_dgrad, tensor_gemm_fprop, tensor_gemm_wgrad,
                      tensor_quantize, bgrad_from_operand, quantize_dbias, mx_quantize_dbias)

__all__ = ["ACC_FAST", "ACC_FULL", "E4M3", "E5M2", "EPI_BIAS", "EPI_BIAS_GELU", "EPI_DGELU", "EPI_DGELU_BGRAD",
           "EPI_NONE", "EXPORTS", "Fp8Error", "Fp8Tensor", "cast_f32", "debug_starve_next_gemm", "device_status",
           "empty_fp8", "gemm_dgrad", "gemm_dgrad_quant", "gemm_fprop", "gemm_wgrad", "grouped_wgrad", "lib", "quantize", "quantize_dual", "scale_ld",
           "status_string", "workspace_size", "Fp8MxTensor", "empty_mx", "mx_gemm_dgrad", "mx_gemm_fprop",
           "mx_gemm_wgrad", "mx_quantize", "mx_sf_bytes", "Fp8TensorScaled", "amax_history_update",
           "empty_tensor_scaled", "tensor_amax", "tensor_gemm_dgrad", "tensor_gemm_fprop", "tensor_gemm_wgrad",
           "tensor_quantize", "bgrad_from_operand", "quantize_dbias", "mx_quantize_dbias"]
