// cast_rule.cuh -- the per-128-block fp8 cast rule, shared by the cast kernels
// and the data-gradient GEMM epilogue that casts its own output, so both give
// the same codes and scales for the same bf16 values.
//
// "Weight gradient kernels for dense and MoE models" casts GEMM operands per
// token with one fp32 scale per 128 elements; the rule (the oracle implements
// it independently):
//   amax = max|x|, inv = fl32(FMAX/amax), scale = fl32(amax/FMAX),
//   q = RNE-saturating fp8(fl32(x * inv)),
// with inv = scale = 1 for a block whose amax is 0 or whose FMAX/amax
// overflows fp32.  IEEE round-to-nearest division and multiplication
// (__fdiv_rn / __fmul_rn, no flush-to-zero).
#pragma once
#include <cfloat>
#include <cstdint>

#include "ptx.cuh"

namespace fp8ll {

template <int FMT>
struct Fp8Fmt;
template <>
struct Fp8Fmt<0> {
    static constexpr float kMax = 448.0f;
    __device__ static uint16_t cvt2(float lo, float hi) { return cvt_e4m3x2(lo, hi); }
};
template <>
struct Fp8Fmt<1> {
    static constexpr float kMax = 57344.0f;
    __device__ static uint16_t cvt2(float lo, float hi) { return cvt_e5m2x2(lo, hi); }
};

template <int FMT>
__device__ __forceinline__ void block_scale(float amax, float& inv, float& scale) {
    inv = 1.0f;
    scale = 1.0f;
    if (amax > 0.0f) {
        const float t = __fdiv_rn(Fp8Fmt<FMT>::kMax, amax);
        if (t <= FLT_MAX) {
            inv = t;
            scale = __fdiv_rn(amax, Fp8Fmt<FMT>::kMax);
        }
    }
}

// two values -> two codes (lo in the low byte) with the block's inv
template <int FMT>
__device__ __forceinline__ uint16_t encode2(float lo, float hi, float inv) {
    return Fp8Fmt<FMT>::cvt2(__fmul_rn(lo, inv), __fmul_rn(hi, inv));
}

}  // namespace fp8ll
