// gemm_fprop.cu -- forward-GEMM instantiations (bf16 out; bias / tanh-GELU epilogues).
#include "gemm_kernel.cuh"

namespace fp8ll {

int launch_gemm_fprop(const TensorMaps& maps, const GemmParams& p, int epi, int fast, cudaStream_t stream,
                      int grid) {
    switch (epi) {
        case kEpiNone:
            return fast ? launch_gemm_impl<kEpiNone, true>(maps, p, stream, grid)
                        : launch_gemm_impl<kEpiNone, false>(maps, p, stream, grid);
        case kEpiBias:
            return fast ? launch_gemm_impl<kEpiBias, true>(maps, p, stream, grid)
                        : launch_gemm_impl<kEpiBias, false>(maps, p, stream, grid);
        case kEpiBiasGelu:
            return fast ? launch_gemm_impl<kEpiBiasGelu, true>(maps, p, stream, grid)
                        : launch_gemm_impl<kEpiBiasGelu, false>(maps, p, stream, grid);
        default:
            return -1;
    }
}

}  // namespace fp8ll
