// common.cuh -- small device helpers shared by the library's kernels.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "ptx.cuh"

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
// Both take a pair of values (the two columns a thread holds of each
// 8-column chunk): the polynomial parts run as packed fp32x2 operations (one
// instruction for both values, each rounded as the scalar operation would be),
// the exponential and the division per value.  With
//   x = clamp(2 sqrt(2/pi) z (1 + 0.044715 z^2), +-80)
//   gelu(z)  = z / (1 + e^-x)
//   gelu'(z) = sp + 2 sqrt(2/pi) z (1 + 3 * 0.044715 z^2) sp sm,  sp = s(x), sm = e^-x sp.

// 2 sqrt(2/pi) z (1 + 0.044715 z^2) for both values, and z^2
__device__ __forceinline__ uint64_t gelu_arg2(uint64_t z, uint64_t& z2) {
    const uint64_t c2 = pack_f32x2(1.5957691216057308f, 1.5957691216057308f);  // 2 sqrt(2/pi)
    const uint64_t one = pack_f32x2(1.0f, 1.0f);
    z2 = mul_f32x2(z, z);
    return mul_f32x2(c2, mul_f32x2(z, fma_f32x2(z2, pack_f32x2(0.044715f, 0.044715f), one)));
}

__device__ __forceinline__ float2 gelu_tanh2(float z0, float z1) {
    uint64_t z2;
    const float2 x = unpack_f32x2(gelu_arg2(pack_f32x2(z0, z1), z2));
    const float x0 = fminf(fmaxf(x.x, -80.0f), 80.0f), x1 = fminf(fmaxf(x.y, -80.0f), 80.0f);
    return make_float2(__fdividef(z0, 1.0f + __expf(-x0)), __fdividef(z1, 1.0f + __expf(-x1)));
}

__device__ __forceinline__ float2 dgelu_tanh2(float z0, float z1) {
    const uint64_t z = pack_f32x2(z0, z1);
    uint64_t z2;
    const float2 x = unpack_f32x2(gelu_arg2(z, z2));
    const float x0 = fminf(fmaxf(x.x, -80.0f), 80.0f), x1 = fminf(fmaxf(x.y, -80.0f), 80.0f);
    const float e0 = __expf(-x0), e1 = __expf(-x1);
    const uint64_t sp = pack_f32x2(__fdividef(1.0f, 1.0f + e0), __fdividef(1.0f, 1.0f + e1));  // s(x)
    const uint64_t sm = mul_f32x2(pack_f32x2(e0, e1), sp);                                      // s(-x)
    const uint64_t c2 = pack_f32x2(1.5957691216057308f, 1.5957691216057308f);
    const uint64_t k3 = pack_f32x2(3.0f * 0.044715f, 3.0f * 0.044715f);
    const uint64_t v = mul_f32x2(mul_f32x2(c2, z), fma_f32x2(z2, k3, pack_f32x2(1.0f, 1.0f)));
    return unpack_f32x2(fma_f32x2(mul_f32x2(v, sp), sm, sp));
}

// Hint that a global cache line will be read soon: fetched into L2 ahead of use.
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

__device__ __forceinline__ void record_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

}  // namespace fp8ll
