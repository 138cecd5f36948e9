// gemm_fprop.cu -- forward-GEMM instantiations (bf16 out; bias / tanh-GELU epilogues).
#include "gemm_kernel.cuh"

namespace fp8ll {

int launch_gemm_fprop(const TensorMaps& maps, const GemmParams& p, int epi, cudaStream_t stream, int grid) {
    switch (epi) {
        case kEpiNone: return launch_gemm_impl<kEpiNone>(maps, p, stream, grid);
        case kEpiBias: return launch_gemm_impl<kEpiBias>(maps, p, stream, grid);
        case kEpiBiasGelu: return launch_gemm_impl<kEpiBiasGelu>(maps, p, stream, grid);
        default: return -1;
    }
}

}  // namespace fp8ll
