// gemm_dgrad.cu -- data-gradient GEMM instantiations (GELU-derivative epilogue,
// optional bias-gradient partial sums) and the bias-gradient finalize kernel.
#include "gemm_kernel.cuh"

namespace fp8ll {

// bgrad[j] = sum over bands b (ascending) of ws[b][j]; one thread per column,
// fixed order, so the result is deterministic.
__global__ void bgrad_finalize_kernel(const float* __restrict__ ws, int64_t num_bands, int64_t N,
                                      float* __restrict__ bgrad) {
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < N;
         j += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float s = 0.0f;
        for (int64_t b = 0; b < num_bands; ++b) s += ws[b * N + j];
        bgrad[j] = s;
    }
}

int launch_bgrad_finalize(const float* ws, int64_t num_bands, int64_t N, float* bgrad, cudaStream_t stream,
                          int num_sms) {
    int64_t blocks = (N + 255) / 256;
    if (blocks > 4LL * num_sms) blocks = 4LL * num_sms;
    if (blocks < 1) blocks = 1;
    bgrad_finalize_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(ws, num_bands, N, bgrad);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_gemm_dgrad(const TensorMaps& maps, const GemmParams& p, int epi, int fast, cudaStream_t stream,
                      int grid) {
    switch (epi) {
        case kEpiDgelu:
            return fast ? launch_gemm_impl<kEpiDgelu, true>(maps, p, stream, grid)
                        : launch_gemm_impl<kEpiDgelu, false>(maps, p, stream, grid);
        case kEpiDgeluBgrad:
            return fast ? launch_gemm_impl<kEpiDgeluBgrad, true>(maps, p, stream, grid)
                        : launch_gemm_impl<kEpiDgeluBgrad, false>(maps, p, stream, grid);
        default:
            return -1;
    }
}

}  // namespace fp8ll
