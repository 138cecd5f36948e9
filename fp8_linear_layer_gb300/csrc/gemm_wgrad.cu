// gemm_wgrad.cu -- weight-gradient GEMM instantiation (fp32 out (+)= C), used
// by both the dense and the k-grouped entry points.
#include "gemm_kernel.cuh"

namespace fp8ll {

int launch_gemm_wgrad(const TensorMaps& maps, const GemmParams& p, cudaStream_t stream, int grid) {
    return launch_gemm_impl<kEpiWgrad>(maps, p, stream, grid);
}

}  // namespace fp8ll
