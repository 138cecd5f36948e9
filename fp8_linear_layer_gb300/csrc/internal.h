// internal.h -- host-side interfaces between the C-ABI layer and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_params.h"

namespace fp8ll {

int launch_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx, int fmt, int transpose, uint8_t* q,
                    float* scale, int64_t sld, cudaStream_t stream, int num_sms);
int launch_quantize_dual(const void* x, int64_t rows, int64_t cols, int64_t ldx, int fmt, uint8_t* q_rows,
                         float* scale_rows, int64_t sld_rows, uint8_t* q_cols, float* scale_cols, int64_t sld_cols,
                         cudaStream_t stream, int num_sms);
// transposed cast (and, with q_rows, the row cast too) of x plus db = column sums of x:
// partials [rows/128][cols] in dpart, then the fixed-order finalize into dbias
int launch_quantize_dbias(const void* x, int64_t rows, int64_t cols, int64_t ldx, int fmt, uint8_t* q_cols,
                          float* scale_cols, int64_t sld_cols, uint8_t* q_rows, float* scale_rows, int64_t sld_rows,
                          float* dpart, float* dbias, cudaStream_t stream, int num_sms);
// MXFP8 transposed cast of x plus db = column sums of x (partials in dpart, then the finalize)
int launch_mx_quantize_dbias(const void* x, int64_t rows, int64_t cols, int64_t ldx, int fmt, uint8_t* q,
                             uint8_t* sf, float* dpart, float* dbias, cudaStream_t stream, int num_sms);
int launch_tensor_amax(const void* x, int64_t rows, int64_t cols, int64_t ldx, float* amax, cudaStream_t stream,
                       int num_sms);
int launch_tensor_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx, int fmt, const float* amax_in,
                           uint8_t* q_rows, uint8_t* q_cols, float* scale, float* amax_out, cudaStream_t stream,
                           int num_sms);
int launch_amax_history(float* hist, int64_t count, int64_t len, const float* amax_new, float* amax_use,
                        cudaStream_t stream);
int launch_operand_rowsum(const uint8_t* q, int64_t ldq, const float* scale, int64_t sld, int fmt, int64_t rows,
                          int64_t K, float* db, int accumulate, cudaStream_t stream, int num_sms);
int64_t mx_sf_groups(int64_t rows);
int launch_mx_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx, int fmt, int transpose, uint8_t* q,
                       uint8_t* sf, cudaStream_t stream, int num_sms);
int launch_cast_f32(const float* x, int64_t n, int fmt, uint8_t* q, cudaStream_t stream, int num_sms);

// GEMM launchers, one per epilogue family (separate translation units).
// The 1x128 GEMM has one promotion schedule: FP8LL_ACC_FAST is accepted by the
// entry points and runs it (every K block meets its own scale pair).
int launch_gemm_fprop(const TensorMaps& maps, const GemmParams& p, int epi, cudaStream_t stream, int grid);
int launch_gemm_dgrad(const TensorMaps& maps, const GemmParams& p, int epi, cudaStream_t stream, int grid);
int launch_gemm_wgrad(const TensorMaps& maps, const GemmParams& p, cudaStream_t stream, int grid);
// The MXFP8 and per-tensor GEMMs run on CTA pairs over 256 x 256 tiles
// (p.num_m_pairs, p.tiles_per_group in pair tiles) and size their own grids.
int launch_gemm_mx(const TensorMaps& maps, const GemmParams& p, int epi, cudaStream_t stream);
int launch_gemm_tensor(const TensorMaps& maps, const GemmParams& p, int epi, cudaStream_t stream);
int launch_bgrad_finalize(const float* ws, int64_t num_bands, int64_t N, float* bgrad, cudaStream_t stream,
                          int num_sms);

}  // namespace fp8ll
