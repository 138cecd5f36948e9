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
// cudaGetSymbolAddress while that device is current and keeps it.  Under lazy
// module loading (the CUDA default) that first lookup is also when the CUDA
// runtime loads this file's module and reserves the 16 MiB: make the first
// call at start-up, before the caller's own allocator takes the device's
// memory and before any stream capture.  The kept address belongs to the
// current CUDA context; after cudaDeviceReset the library must be reloaded.
// All calls share the one array: calls whose kernels overlap on the GPU (for
// example on two streams) race on it.  Nothing in it needs clearing between
// calls: every partial the bias-gradient sum reads is written by the same
// call first.
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
// device, with that device current).  FP8LL_ERR_SCRATCH if the runtime cannot
// provide it (for example: no memory left to load the array's module).
int scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8LL_ERR_LAUNCH;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();  // the failed lookup is reported by the return code, not left pending
            return FP8LL_ERR_SCRATCH;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return FP8LL_OK;
}

}  // namespace

extern "C" int fp8_gemm_dgrad_noalloc(int64_t M, int64_t N, int64_t K, const fp8ll_operand_t* A,
                                      const fp8ll_operand_t* B, const void* aux_bf16, int epi, int acc_mode,
                                      void* out_bf16, float* bgrad, fp8ll_stream_t stream) {
    // without the bias-gradient sums there are no partials: nothing to hold
    if (epi != FP8LL_EPI_DGELU_BGRAD)
        return fp8_gemm_dgrad(M, N, K, A, B, aux_bf16, epi, acc_mode, out_bf16, bgrad, nullptr, 0, stream);
    // validation pass: given no workspace, fp8_gemm_dgrad checks every other
    // argument first and then refuses with FP8LL_ERR_WORKSPACE, launching
    // nothing -- so a bad call gets the same code from both entry points
    int rc = fp8_gemm_dgrad(M, N, K, A, B, aux_bf16, epi, acc_mode, out_bf16, bgrad, nullptr, 0, stream);
    if (rc != FP8LL_ERR_WORKSPACE) return rc;
    if (fp8_workspace_size(M, N) > kNoAllocScratchFloats * sizeof(float))
        return FP8LL_ERR_WORKSPACE;  // the built-in scratch is too small for M x N
    void* scratch = nullptr;
    rc = scratch_for_current_device(&scratch);
    if (rc != FP8LL_OK) return rc;
    return fp8_gemm_dgrad(M, N, K, A, B, aux_bf16, epi, acc_mode, out_bf16, bgrad, scratch,
                          kNoAllocScratchFloats * sizeof(float), stream);
}
