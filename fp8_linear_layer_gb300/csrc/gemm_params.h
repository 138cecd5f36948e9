// gemm_params.h -- what the GEMM kernels receive: tile shape, epilogue kinds,
// the kernel parameter block and the TMA descriptors.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace fp8ll {

constexpr int kMaxGroups = 256;
constexpr int kTileM = 128;  // GEMM output tile rows
constexpr int kTileN = 256;  // GEMM output tile columns

enum EpiKind : int {
    kEpiNone = 0,
    kEpiBias = 1,
    kEpiBiasGelu = 2,
    kEpiDgelu = 3,
    kEpiDgeluBgrad = 4,
    kEpiWgrad = 5,  // fp32 out (+)= C
    kEpiDgeluQuant = 6,  // dgrad: dZ = C * gelu'(Z) -> bf16, plus its e5m2 row cast (codes + 1x128 scales)
};

// One schedulable group of output tiles: all tiles of a group share the same
// K range.  Dense GEMMs have a single group.
struct GroupEntry {
    int32_t kb_start;  // first 128-deep K block (also the scale row index)
    int32_t nkb;       // number of K blocks (0 allowed for zero-filling)
    int32_t out_index; // which M x N output slab the group writes
    int32_t pad;
};

struct GemmParams {
    int32_t M, N;
    int32_t num_m_tiles, num_n_tiles;  // 128-row and 256-column tiles
    int32_t num_m_pairs;               // MXFP8 / per-tensor GEMMs: 256-row tiles of a CTA pair
    int32_t tiles_per_group;
    int32_t num_groups;
    int32_t total_tiles;
    int32_t accumulate;   // wgrad: 1 = out +=, 0 = out =
    int32_t debug_starve; // test hook: producer issues no loads
    int32_t z_tma;        // dgrad: 1 = stored Z tiles staged in shared memory by TMA (maps.z)
    uint32_t idesc;       // tcgen05 instruction descriptor (formats, tile shape)
    uint64_t budget_ns;   // wall-clock budget of each pipeline wait
    void* out;            // bf16 [M][N] (fprop/dgrad) or fp32 [G][M][N] (wgrad)
    void* aux;            // bf16 [M][N]: Z written by fprop BIAS_GELU, read by dgrad
    const void* bias;     // bf16 [N]
    float* workspace;     // fp32 [4 * num_m_tiles][N] bias-gradient partials (one per 32-row band)
    int* status;          // device status word
    const uint8_t* sfa;   // MXFP8: scale atoms of A and B (UE8M0, the MX cast's layout)
    const uint8_t* sfb;
    int64_t sfa_groups;   // MXFP8: 128-row groups per K block of each scale array
    int64_t sfb_groups;
    const float* tsa;     // per-tensor scaling: the one fp32 scale of A and of B
    const float* tsb;
    uint8_t* qout;        // kEpiDgeluQuant: e5m2 codes of the bf16 dZ, [M][N]
    float* qscale;        // kEpiDgeluQuant: their scales, [N/128][qsld]
    int64_t qsld;
    GroupEntry groups[kMaxGroups];
};

struct TensorMaps {
    CUtensorMap a, b, sa, sb;
    CUtensorMap z;  // dgrad with z_tma: Z bf16 [M][N] in 64 x 128 boxes, 128-byte swizzle
};

}  // namespace fp8ll
