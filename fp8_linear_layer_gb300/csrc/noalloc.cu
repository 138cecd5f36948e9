// noalloc.cu -- fp8_gemm_dgrad_noalloc: the data-gradient GEMM with its
// bias-gradient sums, for callers that cannot allocate device memory.
//
// Who needs this: code that runs where cudaMalloc is not available or not
// allowed -- a runtime whose allocator owns all device memory and forbids
// allocations after start-up, a step replayed from a fixed memory plan, or a
// plain C caller with no device allocator of its own.  fp8_gemm_dgrad asks
// such callers for a workspace; this entry point brings its own.
//
// The workspace (one fp32 partial column sum per 32-row band of the output)
// lives in a file-scope __device__ array of kNoAllocScratchFloats floats
// (16 MiB).  Every GPU that loads the library holds that array until the
// process exits.  Host code cannot use the array's name as a device address,
// so the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current and keeps it; make that
// first call before any stream capture.  All calls share the one array: calls
// whose kernels overlap on the GPU (for example on two streams) race on it.
// Nothing in it needs clearing between calls: every partial the bias-gradient
// sum reads is written by the same call first.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "fp8ll.h"

constexpr size_t kNoAllocScratchFloats = size_t(4) << 20;  // 16 MiB of fp32

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

namespace {

std::mutex g_scratch_mutex;
void* g_scratch_ptr[64] = {nullptr};

// Device address of the scratch array on the current device (set up once per
// device, with that device current).
int scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8LL_ERR_LAUNCH;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FP8LL_ERR_LAUNCH;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return FP8LL_OK;
}

}  // namespace

extern "C" int fp8_gemm_dgrad_noalloc(int64_t M, int64_t N, int64_t K, const fp8ll_operand_t* A,
                                      const fp8ll_operand_t* B, const void* aux_bf16, int epi, int acc_mode,
                                      void* out_bf16, float* bgrad, fp8ll_stream_t stream) {
    if (epi == FP8LL_EPI_DGELU_BGRAD && M >= 1 && N >= 1 &&
        fp8_workspace_size(M, N) > kNoAllocScratchFloats * sizeof(float))
        return FP8LL_ERR_WORKSPACE;  // the built-in scratch is too small for M x N
    void* scratch = nullptr;
    if (epi == FP8LL_EPI_DGELU_BGRAD) {
        const int rc = scratch_for_current_device(&scratch);
        if (rc != FP8LL_OK) return rc;
    }
    return fp8_gemm_dgrad(M, N, K, A, B, aux_bf16, epi, acc_mode, out_bf16, bgrad, scratch,
                          scratch ? kNoAllocScratchFloats * sizeof(float) : 0, stream);
}
