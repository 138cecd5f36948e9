// gemm_dgrad.cu -- data-gradient GEMM instantiations (GELU-derivative epilogue,
// optional bias-gradient partial sums) and the bias-gradient finalize kernel.
#include "gemm_kernel.cuh"

namespace fp8ll {

// bgrad[j] = sum over the bands b of ws[b][j].  A CTA of 256 threads covers 32
// columns with 8 threads each: thread s of a column sums bands s, s + 8,
// s + 16, ... in ascending order (independent loads, several in flight), and
// the eight partial sums are added in the order s = 0..7.  A fixed order, so
// the result is deterministic.
constexpr int kFinalizeSplit = 8;

__global__ void __launch_bounds__(256) bgrad_finalize_kernel(const float* __restrict__ ws, int64_t num_bands,
                                                             int64_t N, float* __restrict__ bgrad) {
    __shared__ float part[kFinalizeSplit][32];
    const int cl = threadIdx.x & 31;  // column within the CTA's 32
    const int sl = threadIdx.x >> 5;  // band slice
    for (int64_t j0 = static_cast<int64_t>(blockIdx.x) * 32; j0 < N; j0 += static_cast<int64_t>(gridDim.x) * 32) {
        const int64_t j = j0 + cl;
        float s = 0.0f;
        if (j < N) {
#pragma unroll 8
            for (int64_t b = sl; b < num_bands; b += kFinalizeSplit) s += ws[b * N + j];
        }
        part[sl][cl] = s;
        __syncthreads();
        if (sl == 0 && j < N) {
            float t = part[0][cl];
#pragma unroll
            for (int i = 1; i < kFinalizeSplit; ++i) t += part[i][cl];
            bgrad[j] = t;
        }
        __syncthreads();
    }
}

int launch_bgrad_finalize(const float* ws, int64_t num_bands, int64_t N, float* bgrad, cudaStream_t stream,
                          int num_sms) {
    int64_t blocks = (N + 31) / 32;
    if (blocks > 8LL * num_sms) blocks = 8LL * num_sms;
    if (blocks < 1) blocks = 1;
    bgrad_finalize_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(ws, num_bands, N, bgrad);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_gemm_dgrad(const TensorMaps& maps, const GemmParams& p, int epi, cudaStream_t stream, int grid) {
    switch (epi) {
        case kEpiDgelu: return launch_gemm_impl<kEpiDgelu>(maps, p, stream, grid);
        case kEpiDgeluBgrad: return launch_gemm_impl<kEpiDgeluBgrad>(maps, p, stream, grid);
        case kEpiDgeluQuant: return launch_gemm_impl<kEpiDgeluQuant>(maps, p, stream, grid);
        default: return -1;
    }
}

}  // namespace fp8ll
