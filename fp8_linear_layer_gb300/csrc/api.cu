// api.cu -- the C ABI (include/fp8ll.h): host-side validation, TMA descriptor
// encoding, device checks and kernel launches.  No allocation, no implicit
// synchronization (fp8_get_device_status excepted).
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fp8ll.h"
#include "internal.h"

namespace fp8ll {

// Device status word: kernels record the first pipeline time-out here.
__device__ int g_status_word = 0;

namespace {

constexpr uint64_t kDefaultBudgetNs = 2000000000ull;  // 2 s per pipeline wait

struct DeviceInfo {
    bool checked = false;
    bool supported = false;
    int num_sms = 0;
    int* status = nullptr;
};

std::mutex g_mutex;
DeviceInfo g_devices[64];
std::atomic<int> g_starve_ms{0};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Current device; checks it is sm_103 and caches SM count and status address.
int current_device(DeviceInfo** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8LL_ERR_LAUNCH;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_devices[dev];
    if (!d.checked) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FP8LL_ERR_LAUNCH;
        d.supported = (major == 10 && minor == 3);
        d.num_sms = sms;
        if (d.supported) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return FP8LL_ERR_LAUNCH;
            d.status = static_cast<int*>(p);
        }
        d.checked = true;
    }
    if (!d.supported) return FP8LL_ERR_UNSUPPORTED_DEVICE;
    *out = &d;
    return FP8LL_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_fmt(int f) { return f == FP8LL_E4M3 || f == FP8LL_E5M2; }

// Checks one GEMM operand with `rows` rows and a K extent of `kext` columns.
bool valid_operand(const fp8ll_operand_t* op, int64_t rows, int64_t kext) {
    if (!op || !op->q || !op->scale) return false;
    if (!aligned16(op->q) || !aligned16(op->scale)) return false;
    if (!valid_fmt(op->fmt)) return false;
    if (op->ld_q < kext || op->ld_q % 16 != 0 || op->ld_q >= (1LL << 39)) return false;
    if (op->scale_ld < rows || op->scale_ld % 4 != 0 || op->scale_ld >= (1LL << 36)) return false;
    if (rows < 1 || rows > (1LL << 31) - 1) return false;
    return true;
}

// TMA descriptors for one operand: codes [rows][kext] (row stride ld_q) in
// 128 x box_rows byte boxes with 128-byte swizzle; scales [kext/128][scale_ld]
// in box_rows x 1 boxes.  Out-of-range rows read as zero.
bool encode_operand(const fp8ll_operand_t* op, int64_t rows, int64_t kext, uint32_t box_rows, CUtensorMap* qmap,
                    CUtensorMap* smap) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint32_t estr[2] = {1, 1};
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kext), static_cast<cuuint64_t>(rows)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(op->ld_q)};
        const cuuint32_t box[2] = {128, box_rows};
        if (enc(qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(op->q), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(kext / 128)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(op->scale_ld) * 4};
        const cuuint32_t box[2] = {box_rows, 1};
        if (enc(smap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(op->scale), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

void init_params(GemmParams& p, int64_t M, int64_t N, const fp8ll_operand_t* A, const fp8ll_operand_t* B,
                 const DeviceInfo* dev) {
    std::memset(&p, 0, sizeof(p));
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.num_m_tiles = static_cast<int32_t>((M + kTileM - 1) / kTileM);
    p.num_n_tiles = static_cast<int32_t>((N + kTileN - 1) / kTileN);
    p.tiles_per_group = p.num_m_tiles * p.num_n_tiles;
    // instruction descriptor of kind::f8f6f4 (fmt 0 = e4m3, 1 = e5m2): bits 4-5
    // D format (1 = f32), 7-9 A format, 10-12 B format, 15/16 A/B major (0 = K),
    // 17-22 N >> 3, 24-28 M >> 4
    p.idesc = (1u << 4) | (static_cast<uint32_t>(A->fmt) << 7) | (static_cast<uint32_t>(B->fmt) << 10) |
              ((static_cast<uint32_t>(kTileN) >> 3) << 17) | ((static_cast<uint32_t>(kTileM) >> 4) << 24);
    p.status = dev->status;
    const int starve = g_starve_ms.exchange(0);
    if (starve > 0) {
        p.debug_starve = 1;
        p.budget_ns = static_cast<uint64_t>(starve) * 1000000ull;
    } else {
        p.budget_ns = kDefaultBudgetNs;
    }
}

int grid_for(const GemmParams& p, const DeviceInfo* dev) {
    return p.total_tiles < dev->num_sms ? p.total_tiles : dev->num_sms;
}

// TMA descriptor for the stored pre-activation Z (bf16 [M][N], row stride
// N * 2 bytes, which TMA needs to be a multiple of 16: N % 8 == 0) in boxes
// of 64 columns x 128 rows with 128-byte swizzling; outside the matrix reads
// as zero.
bool encode_z(const void* z, int64_t M, int64_t N, CUtensorMap* zmap) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kTileM)};
    return enc(zmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(z), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool valid_mn(int64_t M, int64_t N) {
    if (M < 1 || N < 1 || M > (1LL << 31) - 1 || N > (1LL << 31) - 1) return false;
    const int64_t tiles = ((M + kTileM - 1) / kTileM) * ((N + kTileN - 1) / kTileN);
    return tiles < (1LL << 30) && M * N < (1LL << 46);
}

// TMA descriptor for MXFP8 codes [rows][kext] (row stride ld_q), 128 x box_rows
// byte boxes with 128-byte swizzle; out-of-range rows read as zero.
bool encode_codes(const uint8_t* q, int64_t ld_q, int64_t rows, int64_t kext, uint32_t box_rows, CUtensorMap* qmap) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kext), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_q)};
    const cuuint32_t box[2] = {128, box_rows};
    return enc(qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(q), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// TMA descriptor for an MXFP8 scale-atom array (512-byte atoms, the MX cast's
// layout) viewed as rows of 128 32-bit words: boxes of `atoms` whole atoms.
bool encode_sf_atoms(const uint8_t* sf, int64_t num_atoms, uint32_t atoms, CUtensorMap* map) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(num_atoms)};
    const cuuint64_t strides[1] = {512};
    const cuuint32_t box[2] = {128, atoms};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t*>(sf), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool valid_mx_operand(const fp8ll_mx_operand_t* op, int64_t rows, int64_t K) {
    if (!op || !op->q || !op->sf || !valid_fmt(op->fmt)) return false;
    if (!aligned16(op->q) || !aligned16(op->sf)) return false;
    if (op->ld_q < K || op->ld_q % 16 != 0) return false;
    if (rows < 1 || rows > (1LL << 31) - 1) return false;
    return true;
}

// shared setup of the three MXFP8 GEMM entry points
int mx_setup(int64_t M, int64_t N, int64_t K, const fp8ll_mx_operand_t* A, const fp8ll_mx_operand_t* B,
             TensorMaps& maps, GemmParams& p, DeviceInfo** dev) {
    if (!valid_mn(M, N) || K < 128 || K % 128 != 0 || K >= (1LL << 36)) return FP8LL_ERR_INVALID_ARG;
    if (!valid_mx_operand(A, M, K) || !valid_mx_operand(B, N, K)) return FP8LL_ERR_INVALID_ARG;
    int rc = current_device(dev);
    if (rc != FP8LL_OK) return rc;
    std::memset(&maps, 0, sizeof(maps));
    // CTA pairs: each CTA loads 128 rows of A and 128 of B's 256 tile rows,
    // its A scale atom and both atoms of B's 256 rows
    const int64_t sfa_groups = mx_sf_groups(M), sfb_groups = mx_sf_groups(N);
    if (!encode_codes(A->q, A->ld_q, M, K, 128, &maps.a) ||
        !encode_codes(B->q, B->ld_q, N, K, kTileN / 2, &maps.b) ||
        !encode_sf_atoms(A->sf, (K / 128) * sfa_groups, 1, &maps.sa) ||
        !encode_sf_atoms(B->sf, (K / 128) * sfb_groups, 2, &maps.sb))
        return FP8LL_ERR_LAUNCH;
    std::memset(&p, 0, sizeof(p));
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.num_m_tiles = static_cast<int32_t>((M + kTileM - 1) / kTileM);
    p.num_n_tiles = static_cast<int32_t>((N + kTileN - 1) / kTileN);
    p.num_m_pairs = static_cast<int32_t>((M + 255) / 256);
    p.tiles_per_group = p.num_m_pairs * p.num_n_tiles;
    p.num_groups = 1;
    p.groups[0] = GroupEntry{0, static_cast<int32_t>(K / 128), 0, 0};
    p.total_tiles = p.tiles_per_group;
    // block-scaled instruction descriptor: formats, N >> 3, UE8M0 scales, M >> 4
    // (the pair's M = 256); the kernel adds the 32-element group id of each MMA
    // for A and B
    p.idesc = (static_cast<uint32_t>(A->fmt) << 7) | (static_cast<uint32_t>(B->fmt) << 10) |
              ((static_cast<uint32_t>(kTileN) >> 3) << 17) | (1u << 23) | ((256u >> 4) << 24);
    p.status = (*dev)->status;
    const int starve = g_starve_ms.exchange(0);
    if (starve > 0) {
        p.debug_starve = 1;
        p.budget_ns = static_cast<uint64_t>(starve) * 1000000ull;
    } else {
        p.budget_ns = kDefaultBudgetNs;
    }
    p.sfa = A->sf;
    p.sfb = B->sf;
    p.sfa_groups = sfa_groups;
    p.sfb_groups = sfb_groups;
    return FP8LL_OK;
}

bool valid_tensor_operand(const fp8ll_tensor_operand_t* op, int64_t rows, int64_t K) {
    if (!op || !op->q || !op->scale || !valid_fmt(op->fmt)) return false;
    if (!aligned16(op->q) || (reinterpret_cast<uintptr_t>(op->scale) & 3u) != 0) return false;
    if (op->ld_q < K || op->ld_q % 16 != 0 || op->ld_q >= (1LL << 39)) return false;
    if (rows < 1 || rows > (1LL << 31) - 1) return false;
    return true;
}

// shared setup of the three per-tensor GEMM entry points
int tensor_setup(int64_t M, int64_t N, int64_t K, const fp8ll_tensor_operand_t* A, const fp8ll_tensor_operand_t* B,
                 TensorMaps& maps, GemmParams& p, DeviceInfo** dev) {
    if (!valid_mn(M, N) || K < 128 || K % 128 != 0 || K >= (1LL << 36)) return FP8LL_ERR_INVALID_ARG;
    if (!valid_tensor_operand(A, M, K) || !valid_tensor_operand(B, N, K)) return FP8LL_ERR_INVALID_ARG;
    int rc = current_device(dev);
    if (rc != FP8LL_OK) return rc;
    std::memset(&maps, 0, sizeof(maps));
    // CTA pairs: each CTA loads 128 rows of A and 128 of B's 256 tile rows
    if (!encode_codes(A->q, A->ld_q, M, K, 128, &maps.a) ||
        !encode_codes(B->q, B->ld_q, N, K, kTileN / 2, &maps.b))
        return FP8LL_ERR_LAUNCH;
    fp8ll_operand_t pa{A->q, A->scale, A->ld_q, 0, A->fmt, 0}, pb{B->q, B->scale, B->ld_q, 0, B->fmt, 0};
    init_params(p, M, N, &pa, &pb, *dev);  // the plain kind::f8f6f4 instruction descriptor
    p.num_m_pairs = static_cast<int32_t>((M + 255) / 256);
    p.tiles_per_group = p.num_m_pairs * p.num_n_tiles;
    p.idesc = (p.idesc & ~(0x1Fu << 24)) | ((256u >> 4) << 24);  // the pair's MMA: M = 256
    p.num_groups = 1;
    p.groups[0] = GroupEntry{0, static_cast<int32_t>(K / 128), 0, 0};
    p.total_tiles = p.tiles_per_group;
    p.tsa = A->scale;
    p.tsb = B->scale;
    return FP8LL_OK;
}

}  // namespace
}  // namespace fp8ll

using namespace fp8ll;

// true when [a, a + na) and [b, b + nb) share a byte
static bool overlaps(const void* a, int64_t na, const void* b, int64_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + static_cast<uintptr_t>(nb) && y < x + static_cast<uintptr_t>(na);
}

extern "C" {

int64_t fp8_scale_ld(int64_t rows) { return rows <= 0 ? 0 : (rows + 3) / 4 * 4; }

int fp8_quantize(const void* x_bf16, int64_t rows, int64_t cols, int64_t ldx, int fmt, int transpose, uint8_t* q,
                 float* scale, int64_t scale_ld, fp8ll_stream_t stream) {
    if (rows < 0 || cols < 0 || !valid_fmt(fmt) || (transpose != 0 && transpose != 1)) return FP8LL_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return FP8LL_OK;
    if (!x_bf16 || !q || !scale || !aligned16(x_bf16) || !aligned16(q) || !aligned16(scale))
        return FP8LL_ERR_INVALID_ARG;
    if (ldx < cols || ldx % 8 != 0 || scale_ld % 4 != 0) return FP8LL_ERR_INVALID_ARG;
    if (rows > (1LL << 31) - 1 || cols > (1LL << 31) - 1) return FP8LL_ERR_INVALID_ARG;
    if (!transpose) {
        if (cols % 128 != 0 || scale_ld < rows) return FP8LL_ERR_INVALID_ARG;
    } else {
        if (rows % 128 != 0 || cols % 8 != 0 || scale_ld < cols) return FP8LL_ERR_INVALID_ARG;
        if (rows / 128 > 65535) return FP8LL_ERR_INVALID_ARG;
    }
    DeviceInfo* dev = nullptr;
    int rc = current_device(&dev);
    if (rc != FP8LL_OK) return rc;
    return launch_quantize(x_bf16, rows, cols, ldx, fmt, transpose, q, scale, scale_ld,
                           reinterpret_cast<cudaStream_t>(stream), dev->num_sms) == 0
               ? FP8LL_OK
               : FP8LL_ERR_LAUNCH;
}

int fp8_quantize_dual(const void* x_bf16, int64_t rows, int64_t cols, int64_t ldx, int fmt, uint8_t* q_rows,
                      float* scale_rows, int64_t scale_ld_rows, uint8_t* q_cols, float* scale_cols,
                      int64_t scale_ld_cols, fp8ll_stream_t stream) {
    if (rows < 0 || cols < 0 || !valid_fmt(fmt)) return FP8LL_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return FP8LL_OK;
    if (!x_bf16 || !q_rows || !scale_rows || !q_cols || !scale_cols) return FP8LL_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(q_rows) || !aligned16(scale_rows) || !aligned16(q_cols) ||
        !aligned16(scale_cols))
        return FP8LL_ERR_INVALID_ARG;
    if (rows > (1LL << 31) - 1 || cols > (1LL << 31) - 1) return FP8LL_ERR_INVALID_ARG;
    if (rows % 128 != 0 || cols % 128 != 0 || rows / 128 > 65535) return FP8LL_ERR_INVALID_ARG;
    if (ldx < cols || ldx % 8 != 0) return FP8LL_ERR_INVALID_ARG;
    if (scale_ld_rows < rows || scale_ld_rows % 4 != 0 || scale_ld_cols < cols || scale_ld_cols % 4 != 0)
        return FP8LL_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    int rc = current_device(&dev);
    if (rc != FP8LL_OK) return rc;
    return launch_quantize_dual(x_bf16, rows, cols, ldx, fmt, q_rows, scale_rows, scale_ld_rows, q_cols, scale_cols,
                                scale_ld_cols, reinterpret_cast<cudaStream_t>(stream), dev->num_sms) == 0
               ? FP8LL_OK
               : FP8LL_ERR_LAUNCH;
}

int fp8_cast_f32(const float* x, int64_t n, int fmt, uint8_t* q, fp8ll_stream_t stream) {
    if (n < 0 || !valid_fmt(fmt)) return FP8LL_ERR_INVALID_ARG;
    if (n == 0) return FP8LL_OK;
    if (!x || !q || !aligned16(x) || !aligned16(q)) return FP8LL_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    int rc = current_device(&dev);
    if (rc != FP8LL_OK) return rc;
    return launch_cast_f32(x, n, fmt, q, reinterpret_cast<cudaStream_t>(stream), dev->num_sms) == 0
               ? FP8LL_OK
               : FP8LL_ERR_LAUNCH;
}

int fp8_gemm_fprop(int64_t M, int64_t N, int64_t K, const fp8ll_operand_t* A, const fp8ll_operand_t* B,
                   const void* bias_bf16, int epi, int acc_mode, void* out_bf16, void* aux_bf16,
                   fp8ll_stream_t stream) {
    if (!valid_mn(M, N) || K < 128 || K % 128 != 0 || K >= (1LL << 36)) return FP8LL_ERR_INVALID_ARG;
    if (epi != FP8LL_EPI_NONE && epi != FP8LL_EPI_BIAS && epi != FP8LL_EPI_BIAS_GELU) return FP8LL_ERR_INVALID_ARG;
    if (acc_mode != FP8LL_ACC_FULL && acc_mode != FP8LL_ACC_FAST) return FP8LL_ERR_INVALID_ARG;
    if (!valid_operand(A, M, K) || !valid_operand(B, N, K)) return FP8LL_ERR_INVALID_ARG;
    if (!out_bf16 || !aligned16(out_bf16)) return FP8LL_ERR_INVALID_ARG;
    if (epi != FP8LL_EPI_NONE && (!bias_bf16 || !aligned16(bias_bf16))) return FP8LL_ERR_INVALID_ARG;
    if (epi == FP8LL_EPI_BIAS_GELU && aux_bf16 && (!aligned16(aux_bf16) || aux_bf16 == out_bf16))
        return FP8LL_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    int rc = current_device(&dev);
    if (rc != FP8LL_OK) return rc;
    TensorMaps maps;
    if (!encode_operand(A, M, K, 128, &maps.a, &maps.sa) || !encode_operand(B, N, K, kTileN, &maps.b, &maps.sb))
        return FP8LL_ERR_LAUNCH;
    GemmParams p;
    init_params(p, M, N, A, B, dev);
    p.num_groups = 1;
    p.groups[0] = GroupEntry{0, static_cast<int32_t>(K / 128), 0, 0};
    p.total_tiles = p.tiles_per_group;
    p.out = out_bf16;
    p.aux = (epi == FP8LL_EPI_BIAS_GELU) ? aux_bf16 : nullptr;
    p.bias = bias_bf16;
    return launch_gemm_fprop(maps, p, epi, reinterpret_cast<cudaStream_t>(stream), grid_for(p, dev)) == 0
               ? FP8LL_OK
               : FP8LL_ERR_LAUNCH;
}

size_t fp8_workspace_size(int64_t M, int64_t N) {
    if (M < 1 || N < 1) return 0;
    return static_cast<size_t>((M + 127) / 128) * 4 * static_cast<size_t>(N) * sizeof(float);
}

int fp8_gemm_dgrad(int64_t M, int64_t N, int64_t K, const fp8ll_operand_t* A, const fp8ll_operand_t* B,
                   const void* aux_bf16, int epi, int acc_mode, void* out_bf16, float* bgrad, void* workspace,
                   size_t workspace_bytes, fp8ll_stream_t stream) {
    if (!valid_mn(M, N) || K < 128 || K % 128 != 0 || K >= (1LL << 36)) return FP8LL_ERR_INVALID_ARG;
    if (epi != FP8LL_EPI_DGELU && epi != FP8LL_EPI_DGELU_BGRAD) return FP8LL_ERR_INVALID_ARG;
    if (acc_mode != FP8LL_ACC_FULL && acc_mode != FP8LL_ACC_FAST) return FP8LL_ERR_INVALID_ARG;
    if (!valid_operand(A, M, K) || !valid_operand(B, N, K)) return FP8LL_ERR_INVALID_ARG;
    if (!out_bf16 || !aligned16(out_bf16) || !aux_bf16 || !aligned16(aux_bf16)) return FP8LL_ERR_INVALID_ARG;
    if (epi == FP8LL_EPI_DGELU_BGRAD) {
        if (!bgrad || !aligned16(bgrad)) return FP8LL_ERR_INVALID_ARG;
        if (!workspace || !aligned16(workspace) || workspace_bytes < fp8_workspace_size(M, N))
            return FP8LL_ERR_WORKSPACE;
    }
    DeviceInfo* dev = nullptr;
    int rc = current_device(&dev);
    if (rc != FP8LL_OK) return rc;
    TensorMaps maps;
    if (!encode_operand(A, M, K, 128, &maps.a, &maps.sa) || !encode_operand(B, N, K, kTileN, &maps.b, &maps.sb))
        return FP8LL_ERR_LAUNCH;
    GemmParams p;
    init_params(p, M, N, A, B, dev);
    p.num_groups = 1;
    p.groups[0] = GroupEntry{0, static_cast<int32_t>(K / 128), 0, 0};
    p.total_tiles = p.tiles_per_group;
    p.out = out_bf16;
    p.aux = const_cast<void*>(aux_bf16);
    p.workspace = static_cast<float*>(workspace);
    // Z tiles go through shared memory by TMA when its rows are 16-byte aligned;
    // otherwise the epilogue reads them from global memory
    std::memset(&maps.z, 0, sizeof(maps.z));
    if (N % 8 == 0) {
        if (!encode_z(aux_bf16, M, N, &maps.z)) return FP8LL_ERR_LAUNCH;
        p.z_tma = 1;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_gemm_dgrad(maps, p, epi, s, grid_for(p, dev)) != 0) return FP8LL_ERR_LAUNCH;
    if (epi == FP8LL_EPI_DGELU_BGRAD) {
        if (launch_bgrad_finalize(static_cast<const float*>(workspace), static_cast<int64_t>(p.num_m_tiles) * 4, N,
                                  bgrad, s, dev->num_sms) != 0)
            return FP8LL_ERR_LAUNCH;
    }
    return FP8LL_OK;
}

int fp8_gemm_dgrad_quant(int64_t M, int64_t N, int64_t K, const fp8ll_operand_t* A, const fp8ll_operand_t* B,
                         const void* aux_bf16, int acc_mode, void* out_bf16, uint8_t* q, float* scale,
                         int64_t scale_ld, fp8ll_stream_t stream) {
    if (!valid_mn(M, N) || K < 128 || K % 128 != 0 || K >= (1LL << 36) || N % 128 != 0) return FP8LL_ERR_INVALID_ARG;
    if (acc_mode != FP8LL_ACC_FULL && acc_mode != FP8LL_ACC_FAST) return FP8LL_ERR_INVALID_ARG;
    if (!valid_operand(A, M, K) || !valid_operand(B, N, K)) return FP8LL_ERR_INVALID_ARG;
    if (!out_bf16 || !aligned16(out_bf16) || !aux_bf16 || !aligned16(aux_bf16)) return FP8LL_ERR_INVALID_ARG;
    if (!q || !aligned16(q) || !scale || !aligned16(scale) || scale_ld < M || scale_ld % 4 != 0)
        return FP8LL_ERR_INVALID_ARG;
    // the codes and scales are written while dZ is written and Z is read
    const int64_t q_bytes = M * N, s_bytes = ((N / 128 - 1) * scale_ld + M) * 4, z_bytes = M * N * 2;
    if (overlaps(q, q_bytes, out_bf16, z_bytes) || overlaps(q, q_bytes, aux_bf16, z_bytes) ||
        overlaps(scale, s_bytes, out_bf16, z_bytes) || overlaps(scale, s_bytes, aux_bf16, z_bytes) ||
        overlaps(q, q_bytes, scale, s_bytes))
        return FP8LL_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    int rc = current_device(&dev);
    if (rc != FP8LL_OK) return rc;
    TensorMaps maps;
    if (!encode_operand(A, M, K, 128, &maps.a, &maps.sa) || !encode_operand(B, N, K, kTileN, &maps.b, &maps.sb))
        return FP8LL_ERR_LAUNCH;
    GemmParams p;
    init_params(p, M, N, A, B, dev);
    p.num_groups = 1;
    p.groups[0] = GroupEntry{0, static_cast<int32_t>(K / 128), 0, 0};
    p.total_tiles = p.tiles_per_group;
    p.out = out_bf16;
    p.aux = const_cast<void*>(aux_bf16);
    p.qout = q;
    p.qscale = scale;
    p.qsld = scale_ld;
    std::memset(&maps.z, 0, sizeof(maps.z));
    if (!encode_z(aux_bf16, M, N, &maps.z)) return FP8LL_ERR_LAUNCH;  // N % 128 == 0: rows 16-byte aligned
    p.z_tma = 1;
    return launch_gemm_dgrad(maps, p, kEpiDgeluQuant, reinterpret_cast<cudaStream_t>(stream), grid_for(p, dev)) == 0
               ? FP8LL_OK
               : FP8LL_ERR_LAUNCH;
}

int fp8_grouped_wgrad(int G, int64_t M, int64_t N, const int64_t* k_sizes, const fp8ll_operand_t* A,
                      const fp8ll_operand_t* B, float* out, int accumulate, int acc_mode, fp8ll_stream_t stream) {
    if (G < 1 || G > kMaxGroups || !k_sizes) return FP8LL_ERR_INVALID_ARG;
    if (!valid_mn(M, N) || (accumulate != 0 && accumulate != 1)) return FP8LL_ERR_INVALID_ARG;
    if (acc_mode != FP8LL_ACC_FULL && acc_mode != FP8LL_ACC_FAST) return FP8LL_ERR_INVALID_ARG;
    if (!out || !aligned16(out)) return FP8LL_ERR_INVALID_ARG;
    int64_t total_k = 0;
    for (int g = 0; g < G; ++g) {
        if (k_sizes[g] < 0 || k_sizes[g] % 128 != 0) return FP8LL_ERR_INVALID_ARG;
        total_k += k_sizes[g];
        if (total_k >= (1LL << 36)) return FP8LL_ERR_INVALID_ARG;
    }
    if (static_cast<int64_t>(G) * M * N >= (1LL << 46)) return FP8LL_ERR_INVALID_ARG;
    if (total_k > 0 && (!valid_operand(A, M, total_k) || !valid_operand(B, N, total_k)))
        return FP8LL_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    int rc = current_device(&dev);
    if (rc != FP8LL_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t slab = static_cast<size_t>(M) * static_cast<size_t>(N) * sizeof(float);
    GemmParams p;
    int ng = 0;
    if (total_k > 0) init_params(p, M, N, A, B, dev);
    // groups with work, longest first (ties keep their order) for load balance
    int order[kMaxGroups];
    for (int g = 0; g < G; ++g) order[g] = g;
    for (int i = 1; i < G; ++i) {
        const int v = order[i];
        int j = i - 1;
        while (j >= 0 && k_sizes[order[j]] < k_sizes[v]) {
            order[j + 1] = order[j];
            --j;
        }
        order[j + 1] = v;
    }
    int64_t offs[kMaxGroups];
    int64_t acc_off = 0;
    for (int g = 0; g < G; ++g) {
        offs[g] = acc_off;
        acc_off += k_sizes[g];
    }
    for (int i = 0; i < G; ++i) {
        const int g = order[i];
        if (k_sizes[g] == 0) {
            // an empty group contributes nothing: keep out_g, or zero it for out =
            if (!accumulate && cudaMemsetAsync(out + static_cast<size_t>(g) * M * N, 0, slab, s) != cudaSuccess)
                return FP8LL_ERR_LAUNCH;
            continue;
        }
        p.groups[ng++] = GroupEntry{static_cast<int32_t>(offs[g] / 128), static_cast<int32_t>(k_sizes[g] / 128), g, 0};
    }
    if (ng == 0) return FP8LL_OK;
    TensorMaps maps;
    if (!encode_operand(A, M, total_k, 128, &maps.a, &maps.sa) ||
        !encode_operand(B, N, total_k, kTileN, &maps.b, &maps.sb))
        return FP8LL_ERR_LAUNCH;
    p.num_groups = ng;
    p.total_tiles = ng * p.tiles_per_group;
    p.out = out;
    p.accumulate = accumulate;
    return launch_gemm_wgrad(maps, p, s, grid_for(p, dev)) == 0 ? FP8LL_OK : FP8LL_ERR_LAUNCH;
}

int fp8_gemm_wgrad(int64_t M, int64_t N, int64_t K, const fp8ll_operand_t* A, const fp8ll_operand_t* B,
                   float* out, int accumulate, int acc_mode, fp8ll_stream_t stream) {
    if (K < 0) return FP8LL_ERR_INVALID_ARG;
    const int64_t ks[1] = {K};
    return fp8_grouped_wgrad(1, M, N, ks, A, B, out, accumulate, acc_mode, stream);
}

int fp8_bgrad_from_operand(int64_t rows, int64_t K, const fp8ll_operand_t* A, float* db, int accumulate,
                           fp8ll_stream_t stream) {
    if (rows < 0 || K < 0 || K % 128 != 0) return FP8LL_ERR_INVALID_ARG;
    if (rows == 0) return FP8LL_OK;
    if (!db || (reinterpret_cast<uintptr_t>(db) & 3u) != 0 || !valid_operand(A, rows, K)) return FP8LL_ERR_INVALID_ARG;
    // the kernel reads codes and scales through the read-only path: db may overlap neither
    const int64_t qbytes = (rows - 1) * A->ld_q + K;
    const int64_t sbytes = K > 0 ? ((K / 128 - 1) * A->scale_ld + rows) * 4 : 0;
    if (overlaps(db, rows * 4, A->q, qbytes) || overlaps(db, rows * 4, A->scale, sbytes)) return FP8LL_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    int rc = current_device(&dev);
    if (rc != FP8LL_OK) return rc;
    return launch_operand_rowsum(A->q, A->ld_q, A->scale, A->scale_ld, A->fmt, rows, K, db, accumulate ? 1 : 0,
                                 reinterpret_cast<cudaStream_t>(stream), dev->num_sms) == 0
               ? FP8LL_OK
               : FP8LL_ERR_LAUNCH;
}

int fp8_quantize_dbias(const void* x_bf16, int64_t rows, int64_t cols, int64_t ldx, int fmt, uint8_t* q_cols,
                       float* scale_cols, int64_t scale_ld_cols, uint8_t* q_rows, float* scale_rows,
                       int64_t scale_ld_rows, float* dbias, void* workspace, size_t workspace_bytes,
                       fp8ll_stream_t stream) {
    if (rows < 0 || cols < 0 || !valid_fmt(fmt)) return FP8LL_ERR_INVALID_ARG;
    if (cols == 0) return FP8LL_OK;
    if (!dbias || (reinterpret_cast<uintptr_t>(dbias) & 3u) != 0 || cols > (1LL << 31) - 1)
        return FP8LL_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    if (rows == 0) {  // a sum over no rows
        int rc = current_device(&dev);
        if (rc != FP8LL_OK) return rc;
        return cudaMemsetAsync(dbias, 0, static_cast<size_t>(cols) * 4, reinterpret_cast<cudaStream_t>(stream)) ==
                       cudaSuccess
                   ? FP8LL_OK
                   : FP8LL_ERR_LAUNCH;
    }
    if (!x_bf16 || !aligned16(x_bf16) || !q_cols || !aligned16(q_cols) || !scale_cols || !aligned16(scale_cols))
        return FP8LL_ERR_INVALID_ARG;
    if (ldx < cols || ldx % 8 != 0 || rows % 128 != 0 || rows / 128 > 65535 || rows > (1LL << 31) - 1)
        return FP8LL_ERR_INVALID_ARG;
    if (cols % 8 != 0 || scale_ld_cols < cols || scale_ld_cols % 4 != 0) return FP8LL_ERR_INVALID_ARG;
    if (q_rows) {
        if (!aligned16(q_rows) || !scale_rows || !aligned16(scale_rows) || cols % 128 != 0 ||
            scale_ld_rows < rows || scale_ld_rows % 4 != 0)
            return FP8LL_ERR_INVALID_ARG;
    }
    const int64_t part_bytes = (rows / 128) * cols * 4;
    if (!workspace || !aligned16(workspace) || static_cast<int64_t>(workspace_bytes) < part_bytes)
        return FP8LL_ERR_WORKSPACE;
    // the cast kernel writes the partials while it reads x and writes the
    // codes and scales, and the finalize reads them while it writes dbias
    const int64_t x_bytes = ((rows - 1) * ldx + cols) * 2;
    const int64_t qc_bytes = cols * rows, sc_bytes = ((rows / 128 - 1) * scale_ld_cols + cols) * 4;
    if (overlaps(dbias, cols * 4, workspace, part_bytes) || overlaps(x_bf16, x_bytes, workspace, part_bytes) ||
        overlaps(q_cols, qc_bytes, workspace, part_bytes) || overlaps(scale_cols, sc_bytes, workspace, part_bytes))
        return FP8LL_ERR_INVALID_ARG;
    if (q_rows) {
        const int64_t qr_bytes = rows * cols, sr_bytes = ((cols / 128 - 1) * scale_ld_rows + rows) * 4;
        if (overlaps(q_rows, qr_bytes, workspace, part_bytes) || overlaps(scale_rows, sr_bytes, workspace, part_bytes))
            return FP8LL_ERR_INVALID_ARG;
    }
    int rc = current_device(&dev);
    if (rc != FP8LL_OK) return rc;
    return launch_quantize_dbias(x_bf16, rows, cols, ldx, fmt, q_cols, scale_cols, scale_ld_cols, q_rows, scale_rows,
                                 scale_ld_rows, static_cast<float*>(workspace), dbias,
                                 reinterpret_cast<cudaStream_t>(stream), dev->num_sms) == 0
               ? FP8LL_OK
               : FP8LL_ERR_LAUNCH;
}

int fp8_mx_quantize_dbias(const void* x_bf16, int64_t rows, int64_t cols, int64_t ldx, int fmt, uint8_t* q,
                          uint8_t* sf, float* dbias, void* workspace, size_t workspace_bytes, fp8ll_stream_t stream) {
    if (rows < 0 || cols < 0 || !valid_fmt(fmt)) return FP8LL_ERR_INVALID_ARG;
    if (cols == 0) return FP8LL_OK;
    if (!dbias || (reinterpret_cast<uintptr_t>(dbias) & 3u) != 0 || cols > (1LL << 31) - 1)
        return FP8LL_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    if (rows == 0) {  // a sum over no rows
        int rc = current_device(&dev);
        if (rc != FP8LL_OK) return rc;
        return cudaMemsetAsync(dbias, 0, static_cast<size_t>(cols) * 4, reinterpret_cast<cudaStream_t>(stream)) ==
                       cudaSuccess
                   ? FP8LL_OK
                   : FP8LL_ERR_LAUNCH;
    }
    if (!x_bf16 || !q || !sf || !aligned16(x_bf16) || !aligned16(q) || !aligned16(sf)) return FP8LL_ERR_INVALID_ARG;
    if (ldx < cols || ldx % 8 != 0 || rows % 128 != 0 || cols % 8 != 0 || rows / 128 > 65535 ||
        rows > (1LL << 31) - 1)
        return FP8LL_ERR_INVALID_ARG;
    const int64_t part_bytes = (rows / 128) * cols * 4;
    if (!workspace || !aligned16(workspace) || static_cast<int64_t>(workspace_bytes) < part_bytes)
        return FP8LL_ERR_WORKSPACE;
    // as fp8_quantize_dbias: the partials may not overlap what the cast reads or writes
    const int64_t x_bytes = ((rows - 1) * ldx + cols) * 2;
    const int64_t sf_bytes = static_cast<int64_t>(fp8_mx_sf_bytes(cols, rows));
    if (overlaps(dbias, cols * 4, workspace, part_bytes) || overlaps(x_bf16, x_bytes, workspace, part_bytes) ||
        overlaps(q, cols * rows, workspace, part_bytes) || overlaps(sf, sf_bytes, workspace, part_bytes))
        return FP8LL_ERR_INVALID_ARG;
    int rc = current_device(&dev);
    if (rc != FP8LL_OK) return rc;
    return launch_mx_quantize_dbias(x_bf16, rows, cols, ldx, fmt, q, sf, static_cast<float*>(workspace), dbias,
                                    reinterpret_cast<cudaStream_t>(stream), dev->num_sms) == 0
               ? FP8LL_OK
               : FP8LL_ERR_LAUNCH;
}

int fp8_get_device_status(fp8ll_stream_t stream) {
    DeviceInfo* dev = nullptr;
    int rc = current_device(&dev);
    if (rc != FP8LL_OK) return rc;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FP8LL_ERR_LAUNCH;
    int v = 0;
    if (cudaMemcpy(&v, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FP8LL_ERR_LAUNCH;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return FP8LL_ERR_LAUNCH;
    }
    return v;
}

const char* fp8_status_string(int code) {
    switch (code) {
        case FP8LL_OK: return "ok";
        case FP8LL_ERR_INVALID_ARG: return "invalid argument";
        case FP8LL_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103)";
        case FP8LL_ERR_LAUNCH: return "CUDA launch or driver error";
        case FP8LL_ERR_TIMEOUT: return "kernel pipeline wait timed out";
        case FP8LL_ERR_WORKSPACE: return "workspace missing or too small";
        case FP8LL_ERR_SCRATCH: return "built-in scratch array unavailable on this device";
        default: return "unknown status";
    }
}

int fp8_debug_starve_next_gemm(int budget_ms) {
    if (budget_ms < 1 || budget_ms > 10000) return FP8LL_ERR_INVALID_ARG;
    g_starve_ms.store(budget_ms);
    return FP8LL_OK;
}

}  // extern "C"

/* ------------------------------------------------------------------ MXFP8 */

extern "C" {

size_t fp8_mx_sf_bytes(int64_t rows, int64_t k) {
    if (rows < 1 || k < 128 || k % 128 != 0) return 0;
    return static_cast<size_t>(k / 128) * static_cast<size_t>(mx_sf_groups(rows)) * 512;
}

int fp8_mx_quantize(const void* x_bf16, int64_t rows, int64_t cols, int64_t ldx, int fmt, int transpose, uint8_t* q,
                    uint8_t* sf, fp8ll_stream_t stream) {
    if (rows < 0 || cols < 0 || !valid_fmt(fmt) || (transpose != 0 && transpose != 1)) return FP8LL_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return FP8LL_OK;
    if (!x_bf16 || !q || !sf || !aligned16(x_bf16) || !aligned16(q) || !aligned16(sf)) return FP8LL_ERR_INVALID_ARG;
    if (ldx < cols || ldx % 8 != 0) return FP8LL_ERR_INVALID_ARG;
    if (rows > (1LL << 31) - 1 || cols > (1LL << 31) - 1) return FP8LL_ERR_INVALID_ARG;
    if (!transpose) {
        if (cols % 128 != 0) return FP8LL_ERR_INVALID_ARG;
    } else {
        if (rows % 128 != 0 || cols % 8 != 0 || rows / 128 > 65535) return FP8LL_ERR_INVALID_ARG;
    }
    DeviceInfo* dev = nullptr;
    int rc = current_device(&dev);
    if (rc != FP8LL_OK) return rc;
    return launch_mx_quantize(x_bf16, rows, cols, ldx, fmt, transpose, q, sf, reinterpret_cast<cudaStream_t>(stream),
                              dev->num_sms) == 0
               ? FP8LL_OK
               : FP8LL_ERR_LAUNCH;
}

int fp8_mx_gemm_fprop(int64_t M, int64_t N, int64_t K, const fp8ll_mx_operand_t* A, const fp8ll_mx_operand_t* B,
                      const void* bias_bf16, int epi, void* out_bf16, void* aux_bf16, fp8ll_stream_t stream) {
    if (epi != FP8LL_EPI_NONE && epi != FP8LL_EPI_BIAS && epi != FP8LL_EPI_BIAS_GELU) return FP8LL_ERR_INVALID_ARG;
    if (!out_bf16 || !aligned16(out_bf16)) return FP8LL_ERR_INVALID_ARG;
    if (epi != FP8LL_EPI_NONE && (!bias_bf16 || !aligned16(bias_bf16))) return FP8LL_ERR_INVALID_ARG;
    if (epi == FP8LL_EPI_BIAS_GELU && aux_bf16 && (!aligned16(aux_bf16) || aux_bf16 == out_bf16))
        return FP8LL_ERR_INVALID_ARG;
    TensorMaps maps;
    GemmParams p;
    DeviceInfo* dev = nullptr;
    int rc = mx_setup(M, N, K, A, B, maps, p, &dev);
    if (rc != FP8LL_OK) return rc;
    p.out = out_bf16;
    p.aux = (epi == FP8LL_EPI_BIAS_GELU) ? aux_bf16 : nullptr;
    p.bias = bias_bf16;
    return launch_gemm_mx(maps, p, epi, reinterpret_cast<cudaStream_t>(stream)) == 0
               ? FP8LL_OK
               : FP8LL_ERR_LAUNCH;
}

int fp8_mx_gemm_dgrad(int64_t M, int64_t N, int64_t K, const fp8ll_mx_operand_t* A, const fp8ll_mx_operand_t* B,
                      const void* aux_bf16, int epi, void* out_bf16, float* bgrad, void* workspace,
                      size_t workspace_bytes, fp8ll_stream_t stream) {
    if (epi != FP8LL_EPI_DGELU && epi != FP8LL_EPI_DGELU_BGRAD) return FP8LL_ERR_INVALID_ARG;
    if (!out_bf16 || !aligned16(out_bf16) || !aux_bf16 || !aligned16(aux_bf16)) return FP8LL_ERR_INVALID_ARG;
    if (epi == FP8LL_EPI_DGELU_BGRAD) {
        if (!bgrad || !aligned16(bgrad)) return FP8LL_ERR_INVALID_ARG;
        if (!workspace || !aligned16(workspace) || workspace_bytes < fp8_workspace_size(M, N))
            return FP8LL_ERR_WORKSPACE;
    }
    TensorMaps maps;
    GemmParams p;
    DeviceInfo* dev = nullptr;
    int rc = mx_setup(M, N, K, A, B, maps, p, &dev);
    if (rc != FP8LL_OK) return rc;
    p.out = out_bf16;
    p.aux = const_cast<void*>(aux_bf16);
    p.workspace = static_cast<float*>(workspace);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_gemm_mx(maps, p, epi, s) != 0) return FP8LL_ERR_LAUNCH;
    if (epi == FP8LL_EPI_DGELU_BGRAD &&
        launch_bgrad_finalize(static_cast<const float*>(workspace), static_cast<int64_t>(p.num_m_tiles) * 4, N, bgrad,
                              s, dev->num_sms) != 0)
        return FP8LL_ERR_LAUNCH;
    return FP8LL_OK;
}

int fp8_mx_gemm_wgrad(int64_t M, int64_t N, int64_t K, const fp8ll_mx_operand_t* A, const fp8ll_mx_operand_t* B,
                      float* out, int accumulate, fp8ll_stream_t stream) {
    if (!out || !aligned16(out) || (accumulate != 0 && accumulate != 1)) return FP8LL_ERR_INVALID_ARG;
    TensorMaps maps;
    GemmParams p;
    DeviceInfo* dev = nullptr;
    int rc = mx_setup(M, N, K, A, B, maps, p, &dev);
    if (rc != FP8LL_OK) return rc;
    p.out = out;
    p.accumulate = accumulate;
    return launch_gemm_mx(maps, p, kEpiWgrad, reinterpret_cast<cudaStream_t>(stream)) == 0
               ? FP8LL_OK
               : FP8LL_ERR_LAUNCH;
}


int fp8_tensor_amax(const void* x_bf16, int64_t rows, int64_t cols, int64_t ldx, float* amax,
                    fp8ll_stream_t stream) {
    if (rows < 0 || cols < 0 || !amax || (reinterpret_cast<uintptr_t>(amax) & 3u) != 0) return FP8LL_ERR_INVALID_ARG;
    if (rows > 0 && cols > 0) {
        if (!x_bf16 || !aligned16(x_bf16) || cols % 8 != 0 || ldx < cols || ldx % 8 != 0)
            return FP8LL_ERR_INVALID_ARG;
    }
    DeviceInfo* dev = nullptr;
    int rc = current_device(&dev);
    if (rc != FP8LL_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (rows == 0 || cols == 0) return cudaMemsetAsync(amax, 0, sizeof(float), s) == cudaSuccess ? FP8LL_OK
                                                                                                  : FP8LL_ERR_LAUNCH;
    return launch_tensor_amax(x_bf16, rows, cols, ldx, amax, s, dev->num_sms) == 0 ? FP8LL_OK : FP8LL_ERR_LAUNCH;
}

int fp8_tensor_quantize(const void* x_bf16, int64_t rows, int64_t cols, int64_t ldx, int fmt, const float* amax_in,
                        uint8_t* q_rows, uint8_t* q_cols, float* scale, float* amax_out, fp8ll_stream_t stream) {
    if (rows < 0 || cols < 0 || !valid_fmt(fmt)) return FP8LL_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return FP8LL_OK;
    if (!x_bf16 || !aligned16(x_bf16) || !amax_in || !scale || (!q_rows && !q_cols)) return FP8LL_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(amax_in) & 3u) != 0 || (reinterpret_cast<uintptr_t>(scale) & 3u) != 0)
        return FP8LL_ERR_INVALID_ARG;
    if (amax_out && ((reinterpret_cast<uintptr_t>(amax_out) & 3u) != 0 || amax_out == amax_in))
        return FP8LL_ERR_INVALID_ARG;
    // the kernels read *amax_in while one thread writes *scale
    if (static_cast<const void*>(scale) == static_cast<const void*>(amax_in) || scale == amax_out)
        return FP8LL_ERR_INVALID_ARG;
    if (rows > (1LL << 31) - 1 || cols > (1LL << 31) - 1 || ldx < cols || ldx % 8 != 0) return FP8LL_ERR_INVALID_ARG;
    if (q_rows && (!aligned16(q_rows) || cols % 16 != 0)) return FP8LL_ERR_INVALID_ARG;
    if (q_cols && (!aligned16(q_cols) || rows % 128 != 0 || cols % 8 != 0 || rows / 128 > 65535))
        return FP8LL_ERR_INVALID_ARG;
    if (q_rows && q_cols && cols % 128 != 0) return FP8LL_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    int rc = current_device(&dev);
    if (rc != FP8LL_OK) return rc;
    return launch_tensor_quantize(x_bf16, rows, cols, ldx, fmt, amax_in, q_rows, q_cols, scale, amax_out,
                                  reinterpret_cast<cudaStream_t>(stream), dev->num_sms) == 0
               ? FP8LL_OK
               : FP8LL_ERR_LAUNCH;
}

int fp8_amax_history_update(float* history, int64_t count, int64_t len, const float* amax_new, float* amax_use,
                            fp8ll_stream_t stream) {
    if (!history || count < 1 || count > (1 << 20) || len < 1 || len > (1 << 20) || !amax_new || !amax_use)
        return FP8LL_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    int rc = current_device(&dev);
    if (rc != FP8LL_OK) return rc;
    return launch_amax_history(history, count, len, amax_new, amax_use, reinterpret_cast<cudaStream_t>(stream)) ==
                   0
               ? FP8LL_OK
               : FP8LL_ERR_LAUNCH;
}

int fp8_tensor_gemm_fprop(int64_t M, int64_t N, int64_t K, const fp8ll_tensor_operand_t* A,
                          const fp8ll_tensor_operand_t* B, const void* bias_bf16, int epi, void* out_bf16,
                          void* aux_bf16, fp8ll_stream_t stream) {
    if (epi != FP8LL_EPI_NONE && epi != FP8LL_EPI_BIAS && epi != FP8LL_EPI_BIAS_GELU) return FP8LL_ERR_INVALID_ARG;
    if (!out_bf16 || !aligned16(out_bf16)) return FP8LL_ERR_INVALID_ARG;
    if (epi != FP8LL_EPI_NONE && (!bias_bf16 || !aligned16(bias_bf16))) return FP8LL_ERR_INVALID_ARG;
    if (epi == FP8LL_EPI_BIAS_GELU && aux_bf16 && (!aligned16(aux_bf16) || aux_bf16 == out_bf16))
        return FP8LL_ERR_INVALID_ARG;
    TensorMaps maps;
    GemmParams p;
    DeviceInfo* dev = nullptr;
    int rc = tensor_setup(M, N, K, A, B, maps, p, &dev);
    if (rc != FP8LL_OK) return rc;
    p.out = out_bf16;
    p.aux = (epi == FP8LL_EPI_BIAS_GELU) ? aux_bf16 : nullptr;
    p.bias = bias_bf16;
    return launch_gemm_tensor(maps, p, epi, reinterpret_cast<cudaStream_t>(stream)) == 0
               ? FP8LL_OK
               : FP8LL_ERR_LAUNCH;
}

int fp8_tensor_gemm_dgrad(int64_t M, int64_t N, int64_t K, const fp8ll_tensor_operand_t* A,
                          const fp8ll_tensor_operand_t* B, const void* aux_bf16, int epi, void* out_bf16, float* bgrad,
                          void* workspace, size_t workspace_bytes, fp8ll_stream_t stream) {
    if (epi != FP8LL_EPI_DGELU && epi != FP8LL_EPI_DGELU_BGRAD) return FP8LL_ERR_INVALID_ARG;
    if (!out_bf16 || !aligned16(out_bf16) || !aux_bf16 || !aligned16(aux_bf16)) return FP8LL_ERR_INVALID_ARG;
    if (epi == FP8LL_EPI_DGELU_BGRAD) {
        if (!bgrad || !aligned16(bgrad)) return FP8LL_ERR_INVALID_ARG;
        if (!workspace || !aligned16(workspace) || workspace_bytes < fp8_workspace_size(M, N))
            return FP8LL_ERR_WORKSPACE;
    }
    TensorMaps maps;
    GemmParams p;
    DeviceInfo* dev = nullptr;
    int rc = tensor_setup(M, N, K, A, B, maps, p, &dev);
    if (rc != FP8LL_OK) return rc;
    p.out = out_bf16;
    p.aux = const_cast<void*>(aux_bf16);
    p.workspace = static_cast<float*>(workspace);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_gemm_tensor(maps, p, epi, s) != 0) return FP8LL_ERR_LAUNCH;
    if (epi == FP8LL_EPI_DGELU_BGRAD &&
        launch_bgrad_finalize(static_cast<const float*>(workspace), static_cast<int64_t>(p.num_m_tiles) * 4, N, bgrad,
                              s, dev->num_sms) != 0)
        return FP8LL_ERR_LAUNCH;
    return FP8LL_OK;
}

int fp8_tensor_gemm_wgrad(int64_t M, int64_t N, int64_t K, const fp8ll_tensor_operand_t* A,
                          const fp8ll_tensor_operand_t* B, float* out, int accumulate, fp8ll_stream_t stream) {
    if (!out || !aligned16(out) || (accumulate != 0 && accumulate != 1)) return FP8LL_ERR_INVALID_ARG;
    TensorMaps maps;
    GemmParams p;
    DeviceInfo* dev = nullptr;
    int rc = tensor_setup(M, N, K, A, B, maps, p, &dev);
    if (rc != FP8LL_OK) return rc;
    p.out = out;
    p.accumulate = accumulate;
    return launch_gemm_tensor(maps, p, kEpiWgrad, reinterpret_cast<cudaStream_t>(stream)) == 0
               ? FP8LL_OK
               : FP8LL_ERR_LAUNCH;
}

}  // extern "C"
