// common.cuh -- small device helpers shared by the library's kernels.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

namespace fp8ll {

constexpr int kStatusTimeout = -4;  // FP8LL_ERR_TIMEOUT

__device__ __forceinline__ float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t packed) { return __uint_as_float(packed & 0xFFFF0000u); }

// two fp32 -> packed bf16x2 (round to nearest even); `lo` in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// tanh-form GELU and its derivative ("Replaced cublasLt calls with rocblas
// gemm + 6 manually crafted epilogues": GELU epilogue in the forward pass,
// its derivative in the backward pass), evaluated in fp32.
__device__ __forceinline__ float gelu_tanh(float z) {
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    const float u = c * (z + 0.044715f * z * z * z);
    return 0.5f * z * (1.0f + tanhf(u));
}

__device__ __forceinline__ float dgelu_tanh(float z) {
    const float c = 0.7978845608028654f;
    const float z2 = z * z;
    const float t = tanhf(c * (z + 0.044715f * z2 * z));
    return 0.5f * (1.0f + t) + 0.5f * z * (1.0f - t * t) * c * (1.0f + 3.0f * 0.044715f * z2);
}

__device__ __forceinline__ void record_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

}  // namespace fp8ll
