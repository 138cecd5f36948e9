// gemm_wgrad.cu -- weight-gradient GEMM instantiations (fp32 out (+)= C), used
// by both the dense and the k-grouped entry points.
#include "gemm_kernel.cuh"

namespace fp8ll {

int launch_gemm_wgrad(const TensorMaps& maps, const GemmParams& p, int fast, cudaStream_t stream, int grid) {
    return fast ? launch_gemm_impl<kEpiWgrad, true>(maps, p, stream, grid)
                : launch_gemm_impl<kEpiWgrad, false>(maps, p, stream, grid);
}

}  // namespace fp8ll
