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
//   gelu(z)  = 0.5 z (1 + tanh(u)),  u = sqrt(2/pi) (z + 0.044715 z^3)
//   gelu'(z) = 0.5 (1 + tanh u) + 0.5 z (1 - tanh^2 u) sqrt(2/pi) (1 + 3 * 0.044715 z^2)
// written with the logistic identities 0.5 (1 + tanh u) = s(2u) and
// 1 - tanh^2 u = 4 s(2u) s(-2u), s(x) = 1 / (1 + e^-x): the same functions,
// but without the cancellation of 1 + tanh u for large negative z, so both
// keep their relative accuracy everywhere.  2u is clamped to +-80, where s is
// already 0 / 1 to fp32 precision relative to the other term.  The
// exponential is the fast intrinsic (documented error 2 + 1.173 |x| ulp, at
// most ~96 ulp = 6e-6 relative at the clamp) and the divisions the
// approximate fp32 divide (2 ulp): the results are rounded to bf16, whose
// half-ulp is 2e-3 relative, so the evaluation error stays far below the
// output's own rounding.
__device__ __forceinline__ float gelu_tanh(float z) {
    const float c2 = 1.5957691216057308f;  // 2 sqrt(2/pi)
    const float x = fminf(fmaxf(c2 * (z + 0.044715f * z * z * z), -80.0f), 80.0f);
    return __fdividef(z, 1.0f + __expf(-x));
}

__device__ __forceinline__ float dgelu_tanh(float z) {
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    const float z2 = z * z;
    const float x = fminf(fmaxf(2.0f * c * (z + 0.044715f * z2 * z), -80.0f), 80.0f);
    const float e = __expf(-x);
    const float sp = __fdividef(1.0f, 1.0f + e);  // s(2u)
    const float sm = e * sp;                      // s(-2u)
    return sp + 2.0f * z * c * (1.0f + 3.0f * 0.044715f * z2) * sp * sm;
}

// Hint that a global cache line will be read soon: fetched into L2 ahead of use.
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

__device__ __forceinline__ void record_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

}  // namespace fp8ll
