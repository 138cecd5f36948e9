// gemm_kernel.cuh -- persistent block-scaled FP8 GEMM for sm_103a (tcgen05 + TMA + TMEM).
//
// Computes, for every output tile, C[i][j] = sum_kb sA[kb][i] sB[kb][j] P_kb[i][j]
// with P_kb[i][j] = sum_{k in block kb} qA[i][k] qB[j][k] (raw fp8 products,
// fp32 in TMEM), i.e. the 1x128 block-scaled "nt" GEMM of "Weight gradient
// kernels for dense and MoE models", then applies one of the fused epilogues
// of "Replaced cublasLt calls with rocblas gemm + 6 manually crafted
// epilogues" (bias, tanh-GELU, GELU derivative, bias-gradient column sums) or
// the fp32 weight-gradient read-modify-write (out += C).
//
// CTA = 3 warpgroups (12 warps), one CTA per SM, persistent over a
// rasterized tile list of 128 x 256 output tiles:
//   warp 0      TMA producer: operand tiles (128 x 128 B of A, 256 x 128 B of
//               B, 128-byte swizzle) into a 3-stage ring, block scales into
//               an 8-stage ring (more operand stages measured slower).
//   warp 1      TMEM owner and MMA issuer: per K block, 4 x tcgen05.mma
//               (M=128, N=256, K=32, kind::f8f6f4) into one of two TMEM
//               accumulators (2 x 256 fp32 columns), so the MMAs of block
//               k+1 run while block k is promoted.  An N=256 MMA does twice
//               the work of an N=128 one for the same A operand read, and
//               the tensor core only reaches its full rate at this width.
//   warp 2      dgrad only: TMA loader of the stored pre-activation tile Z
//               (128 x 256 bf16, four 64-column boxes, 128-byte swizzle) into
//               a one-slot shared-memory buffer, issued as soon as the previous
//               tile's epilogue has released it, so that it lands during the
//               K loop instead of being fetched by the epilogue.
//   warp 3      idle (completes the first warpgroup).
//   warps 4-11  promotion + epilogue, two warpgroups of 128 columns each:
//               warp w reads TMEM lanes 32*(w%4)..+31 (its rows) in the
//               16x256b fragment shape, so a thread holds four rows x two
//               columns of every 8-column chunk.  Per K block it loads its raw
//               fp32 partial sums with four pairs of 16-lane loads (32
//               columns each: larger loads cost the register allocator extra
//               moves), hands the buffer back to the MMA warp after the last
//               pair and adds
//               sA*sB*P into a 128-element fp32 register accumulator
//               ("promotion") with packed fp32x2 multiplies and fmas.  One
//               8-byte column-scale load serves eight elements: the scale
//               loads draw on shared-memory bandwidth, which the tensor
//               core's operand reads need as well.
// Registers: launched at kLaunchRegs per thread (the most 384 threads can
// have), the first warpgroup gives registers back (setmaxnreg.dec to
// kRegsCtrl) and the two epilogue warpgroups take them (setmaxnreg.inc to
// kRegsEpi); 128 * kRegsCtrl + 256 * kRegsEpi <= 384 * kLaunchRegs.  The host
// refuses to launch if the compiled kernel's register count differs from
// kLaunchRegs, so the split can never ask for more than the pool.
#pragma once
#include <cstdint>

#include "cast_rule.cuh"
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fp8ll {

constexpr int kBM = kTileM;
constexpr int kBN = kTileN;
constexpr int kBK = 128;  // K bytes per stage == one scale block
constexpr int kStages = 3;
constexpr int kSStages = 8;
constexpr int kEpiGroups = 2;               // epilogue warpgroups
constexpr int kEpiWarps = 4 * kEpiGroups;
constexpr int kFirstEpiWarp = 4;
constexpr int kThreads = 128 + 32 * kEpiWarps;
constexpr int kLaunchRegs = 168;
constexpr int kRegsCtrl = 40;
constexpr int kRegsEpi = 232;
static_assert(128 * kRegsCtrl + 128 * kEpiGroups * kRegsEpi <= kThreads * kLaunchRegs,
              "register split exceeds the pool");
constexpr int kHalfN = kBN / kEpiGroups;  // columns per epilogue thread (128)
static_assert(kHalfN == 128, "four 16x256b.x4 TMEM load pairs per thread and K block");
constexpr int kNumAcc = 2;               // TMEM accumulator buffers
constexpr uint32_t kTmemCols = 512;      // kNumAcc * kBN, a power of two
static_assert(kNumAcc * kBN <= 512, "TMEM capacity");
constexpr int kRasterM = 16;

struct __align__(1024) SmemLayout {
    uint8_t a[kStages][kBM * kBK];
    uint8_t b[kStages][kBN * kBK];
    float sa[kSStages][kBM];
    float sb[kSStages][kBN];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t sfull[kSStages];
    uint64_t sempty[kSStages];
    uint64_t acc_full[kNumAcc];
    uint64_t acc_empty[kNumAcc];
    uint64_t zfull, zempty;
    uint64_t drain;
    uint32_t tmem_base;
};
// The dgrad kernels add the Z tile buffer right after the layout (1024-byte
// aligned, as 128-byte swizzling needs): four boxes of 128 rows x 64 columns.
constexpr int kZBoxCols = 64;
constexpr uint32_t kZBoxBytes = kBM * kZBoxCols * 2;
constexpr uint32_t kZBytes = kBM * kBN * 2;
static_assert(sizeof(SmemLayout) % 1024 == 0, "Z buffer alignment");

template <int EPI>
constexpr bool uses_z() {
    return EPI == kEpiDgelu || EPI == kEpiDgeluBgrad || EPI == kEpiDgeluQuant;
}
template <int EPI>
constexpr size_t smem_bytes() {
    return sizeof(SmemLayout) + (uses_z<EPI>() ? kZBytes : 0) + 1024;
}
static_assert(smem_bytes<kEpiDgelu>() <= 232448, "shared memory budget");

template <int N>
__device__ __forceinline__ void ring_advance(int& idx, uint32_t& phase) {
    if (++idx == N) {
        idx = 0;
        phase ^= 1u;
    }
}

// tile index -> (group, m tile, n tile); within a group, bands of kRasterM
// row-tiles are walked column by column so that concurrently running CTAs
// share operand rows in L2.
__device__ __forceinline__ void decode_tile(const GemmParams& p, int t, int& g, int& mt, int& nt) {
    g = t / p.tiles_per_group;
    const int local = t - g * p.tiles_per_group;
    const int band_tiles = kRasterM * p.num_n_tiles;
    const int band = local / band_tiles;
    const int first_m = band * kRasterM;
    const int rem_m = p.num_m_tiles - first_m;
    const int bm = rem_m < kRasterM ? rem_m : kRasterM;
    const int r = local - band * band_tiles;
    mt = first_m + r % bm;
    nt = r / bm;
}

// ------------------------------------------------------------------ stores
//
// After the promotion a thread holds the 16x256b TMEM fragment of its warp:
// rows row0 + 8r (r = 0..3) and column pairs col0 + 8c + {0, 1} (c = 0..15),
// packed as acc[4c + r] (even column in the low half), where
// row0 = m0 + 32 * quadrant + lane / 4 and col0 = n0 + 128 * half + 2 * (lane % 4).

constexpr int kChunks = kHalfN / 8;  // 8-column chunks per thread (16)

__device__ __forceinline__ void red_add_v2(float* addr, float a, float b) {
    asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(addr), "f"(a), "f"(b) : "memory");
}

// wgrad: out (+)= acc, fp32.  out += acc is a single fp32 add per element,
// done in L2 by a vector reduction (no load round trip; each element receives
// exactly one add per call, so the result is deterministic).  16-byte
// reductions when rows are 16-byte aligned, 8-byte ones otherwise.
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ void store_wgrad(const GemmParams& p, int out_index, int row0, int col0,
                                            const uint64_t (&acc)[4 * kChunks]) {
    if ((p.N & 3) == 0) {
        // rows 16-byte aligned: neighbouring lanes of a quad swap one column
        // pair so that each holds four consecutive columns of one chunk of a
        // chunk pair (even lane: the first chunk, odd lane: the second) and
        // adds them with one 16-byte reduction
        const int cq = (col0 >> 1) & 3;
        const bool odd = (cq & 1) != 0;
        const int cb = col0 - 2 * (cq & 1);  // first column of the lane pair
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int row = row0 + 8 * r;
            float* orow = static_cast<float*>(p.out) + (static_cast<int64_t>(out_index) * p.M + row) * p.N;
#pragma unroll
            for (int c = 0; c < kChunks; c += 2) {
                const uint64_t mine = odd ? acc[4 * (c + 1) + r] : acc[4 * c + r];
                const uint64_t recv = __shfl_xor_sync(0xffffffffu, odd ? acc[4 * c + r] : acc[4 * (c + 1) + r], 1);
                const float2 lo = unpack_f32x2(odd ? recv : mine), hi = unpack_f32x2(odd ? mine : recv);
                const int col = cb + 8 * (c + (odd ? 1 : 0));
                if (row >= p.M || col >= p.N) continue;
                if (p.accumulate)
                    red_add_v4(orow + col, lo.x, lo.y, hi.x, hi.y);
                else
                    *reinterpret_cast<float4*>(orow + col) = make_float4(lo.x, lo.y, hi.x, hi.y);
            }
        }
        return;
    }
    const bool pairs = (p.N & 1) == 0;  // column pairs are 8-byte aligned
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int row = row0 + 8 * r;
        if (row >= p.M) continue;
        float* orow = static_cast<float*>(p.out) + (static_cast<int64_t>(out_index) * p.M + row) * p.N;
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
            const int col = col0 + 8 * c;
            const float2 v = unpack_f32x2(acc[4 * c + r]);
            if (pairs) {
                if (col < p.N) {
                    if (p.accumulate)
                        red_add_v2(orow + col, v.x, v.y);
                    else
                        *reinterpret_cast<float2*>(orow + col) = v;
                }
            } else {
                if (col < p.N) orow[col] = (p.accumulate ? orow[col] : 0.0f) + v.x;
                if (col + 1 < p.N) orow[col + 1] = (p.accumulate ? orow[col + 1] : 0.0f) + v.y;
            }
        }
    }
}

// 4 x 4 transpose of 32-bit words among the four lanes of a quad (lanes that
// differ in bits 0-1): on entry a[j] is this lane's word j; on exit a[j] is
// word (lane % 4) of lane j.  Two butterfly stages, two shuffles each.
__device__ __forceinline__ void quad_transpose(uint32_t (&a)[4], int cq) {
    const bool odd = (cq & 1) != 0;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, odd ? a[2 * q] : a[2 * q + 1], 1);
        if (odd)
            a[2 * q] = recv;
        else
            a[2 * q + 1] = recv;
    }
    const bool hi = (cq & 2) != 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, hi ? a[j] : a[2 + j], 2);
        if (hi)
            a[j] = recv;
        else
            a[2 + j] = recv;
    }
}

// fprop: Z = acc + bias[j]; Y = gelu(Z) or Z; bf16 out (+ bf16 aux Z).
// Each chunk's eight values are computed without branches (rows or columns
// outside the matrix compute on zeros) so that their independent GELU
// evaluations overlap; only the memory accesses are guarded.
template <int EPI>
__device__ __forceinline__ void store_fprop(const GemmParams& p, int row0, int col0,
                                            const uint64_t (&acc)[4 * kChunks]) {
    const bool pairs = (p.N & 1) == 0;
    uint16_t* out = static_cast<uint16_t*>(p.out);
    uint16_t* aux = (EPI == kEpiBiasGelu) ? static_cast<uint16_t*>(p.aux) : nullptr;
    const uint16_t* bias = static_cast<const uint16_t*>(p.bias);
    // the bias pairs of all chunks first, so that their loads are in flight together
    uint32_t bw[kChunks];
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        const int col = col0 + 8 * c;
        bw[c] = 0u;
        if (EPI != kEpiNone && col < p.N) {
            if (pairs)
                bw[c] = __ldg(reinterpret_cast<const unsigned int*>(bias + col));
            else
                bw[c] = static_cast<uint32_t>(bias[col]) |
                        (col + 1 < p.N ? static_cast<uint32_t>(bias[col + 1]) << 16 : 0u);
        }
    }
    if ((p.N & 7) == 0) {
        // rows 16-byte aligned: the quad's four lanes swap words so that each
        // holds eight consecutive columns of one chunk and stores them as one
        // 16-byte vector (a warp store then covers 64 contiguous bytes of each
        // of its eight rows)
        const int cq = (col0 >> 1) & 3;
        const int cbase = col0 - 2 * cq;
#pragma unroll
        for (int g = 0; g < kChunks / 4; ++g) {
            uint32_t yw[4][4], zw[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = 4 * g + j;
                const float b0 = bf16_lo(bw[c]), b1 = bf16_hi(bw[c]);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float2 a = unpack_f32x2(acc[4 * c + r]);
                    const float z0 = a.x + b0, z1 = a.y + b1;
                    const float2 y = (EPI == kEpiBiasGelu) ? gelu_tanh2(z0, z1) : make_float2(z0, z1);
                    yw[r][j] = pack_bf16x2(y.x, y.y);
                    zw[r][j] = pack_bf16x2(z0, z1);
                }
            }
            const int col = cbase + 8 * (4 * g + cq);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                quad_transpose(yw[r], cq);
                if (aux) quad_transpose(zw[r], cq);
                const int row = row0 + 8 * r;
                if (row >= p.M || col >= p.N) continue;
                const int64_t off = static_cast<int64_t>(row) * p.N + col;
                *reinterpret_cast<uint4*>(out + off) = make_uint4(yw[r][0], yw[r][1], yw[r][2], yw[r][3]);
                if (aux) *reinterpret_cast<uint4*>(aux + off) = make_uint4(zw[r][0], zw[r][1], zw[r][2], zw[r][3]);
            }
        }
        return;
    }
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        const int col = col0 + 8 * c;
        const bool one = col < p.N, two = col + 1 < p.N;
        const float b0 = bf16_lo(bw[c]), b1 = bf16_hi(bw[c]);
        uint32_t yw[4], zw[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float2 a = unpack_f32x2(acc[4 * c + r]);
            const float z0 = a.x + b0, z1 = a.y + b1;
            const float2 y = (EPI == kEpiBiasGelu) ? gelu_tanh2(z0, z1) : make_float2(z0, z1);
            yw[r] = pack_bf16x2(y.x, y.y);
            zw[r] = pack_bf16x2(z0, z1);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int row = row0 + 8 * r;
            if (row >= p.M || !one) continue;
            const int64_t off = static_cast<int64_t>(row) * p.N + col;
            if (pairs) {
                *reinterpret_cast<uint32_t*>(out + off) = yw[r];
                if (aux) *reinterpret_cast<uint32_t*>(aux + off) = zw[r];
            } else {
                out[off] = static_cast<uint16_t>(yw[r] & 0xFFFFu);
                if (aux) aux[off] = static_cast<uint16_t>(zw[r] & 0xFFFFu);
                if (two) {
                    out[off + 1] = static_cast<uint16_t>(yw[r] >> 16);
                    if (aux) aux[off + 1] = static_cast<uint16_t>(zw[r] >> 16);
                }
            }
        }
    }
}

// dgrad: dZ = acc * gelu'(Z) -> bf16 out.  With BGRAD the fp32 dZ of each
// column (zero outside the matrix) is summed over the warp's 32 rows -- the
// thread's four rows first, then across the eight lanes that hold the same
// columns (lane xor 4, 8, 16), a fixed order, so results are deterministic --
// and the sums go to the workspace band of this warp.  The cross-lane step is
// a reduce-scatter after the last chunk: each of its three stages keeps half
// of the thread's (chunk, column) sums and adds the partner lane's copy of
// them (28 shuffles per thread instead of 96 for a butterfly per chunk), and
// every lane ends with four finished sums to store.
//
// The stored pre-activations come from one of two places.  ZSMEM: the tile's
// Z was staged in shared memory by TMA (zs = the 128 x 256 tile as four
// 64-column boxes with 128-byte swizzling; zeros outside the matrix).  Row r
// of a box is 128 bytes at r * 128, and its 16-byte chunk j sits at
// (j ^ (r % 8)) * 16: the eight rows and four column pairs that one load
// instruction of a warp touches fall in 32 distinct banks.  Otherwise (rows
// of Z not 16-byte aligned) Z is read from global memory.  Either way one
// chunk (4 bf16 pairs) is read at a time, the next chunk's loads in flight
// while the current one is computed (reading the staged chunk just before
// its use measured 3% slower).
constexpr int kZGroup = 1;
static_assert(kZGroup == 1, "Z is read one chunk at a time");

__device__ __forceinline__ void load_z_group(const GemmParams& p, const uint16_t* zp, bool pairs, int row0, int col0,
                                             int c0, uint32_t (&zw)[4 * kZGroup]) {
#pragma unroll
    for (int i = 0; i < kZGroup; ++i) {
        const int col = col0 + 8 * (c0 + i);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int row = row0 + 8 * r;
            uint32_t w = 0u;
            if (row < p.M && col < p.N) {
                const int64_t off = static_cast<int64_t>(row) * p.N + col;
                if (pairs)
                    w = *reinterpret_cast<const uint32_t*>(zp + off);
                else
                    w = static_cast<uint32_t>(zp[off]) |
                        (col + 1 < p.N ? static_cast<uint32_t>(zp[off + 1]) << 16 : 0u);
            }
            zw[4 * i + r] = w;
        }
    }
}

// Z words of chunk c (rows row0 + 8r) from the staged tile; zrow = the
// thread's first row in its half's first box plus 4 * (lane % 4), g8 = row % 8.
__device__ __forceinline__ void load_z_smem(const uint8_t* zrow, int g8, int c, uint32_t (&zw)[4]) {
    const uint8_t* z = zrow + (c >> 3) * kZBoxBytes + (((c & 7) ^ g8) << 4);
#pragma unroll
    for (int r = 0; r < 4; ++r) zw[r] = *reinterpret_cast<const uint32_t*>(z + r * 8 * 128);
}

template <bool BGRAD, bool ZSMEM>
__device__ __forceinline__ void store_dgrad(const GemmParams& p, int row0, int col0,
                                            const uint64_t (&acc)[4 * kChunks], float* band, int lane,
                                            const uint8_t* zrow) {
    const bool pairs = (p.N & 1) == 0;
    uint16_t* out = static_cast<uint16_t*>(p.out);
    const uint16_t* zp = static_cast<const uint16_t*>(p.aux);
    const int g8 = lane >> 2;
    float cs[2 * kChunks];  // BGRAD: column sums over the thread's four rows, per (chunk, column)
    // each chunk's Z words are read one chunk ahead of their use
    uint32_t zcur[4 * kZGroup], znext[4 * kZGroup];
    if (ZSMEM)
        load_z_smem(zrow, g8, 0, zcur);
    else
        load_z_group(p, zp, pairs, row0, col0, 0, zcur);
#pragma unroll
    for (int c0 = 0; c0 < kChunks; c0 += kZGroup) {
        if (c0 + kZGroup < kChunks) {
            if (ZSMEM)
                load_z_smem(zrow, g8, c0 + kZGroup, znext);
            else
                load_z_group(p, zp, pairs, row0, col0, c0 + kZGroup, znext);
        }
#pragma unroll
        for (int i = 0; i < kZGroup; ++i) {
            const int c = c0 + i;
            const int col = col0 + 8 * c;
            const bool one = col < p.N, two = col + 1 < p.N;
            // all eight values first, without branches (outside the matrix the
            // stored pre-activation reads as zero and the value is masked below)
            float d[4][2];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float2 a = unpack_f32x2(acc[4 * c + r]);
                const float2 gd = dgelu_tanh2(bf16_lo(zcur[4 * i + r]), bf16_hi(zcur[4 * i + r]));
                d[r][0] = a.x * gd.x;
                d[r][1] = a.y * gd.y;
            }
            float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int row = row0 + 8 * r;
                const bool ok = row < p.M && one;
                s0 += ok ? d[r][0] : 0.0f;
                s1 += (ok && two) ? d[r][1] : 0.0f;
                if (!ok) continue;
                const int64_t off = static_cast<int64_t>(row) * p.N + col;
                if (pairs) {
                    *reinterpret_cast<uint32_t*>(out + off) = pack_bf16x2(d[r][0], d[r][1]);
                } else {
                    out[off] = static_cast<uint16_t>(pack_bf16x2(d[r][0], 0.0f) & 0xFFFFu);
                    if (two) out[off + 1] = static_cast<uint16_t>(pack_bf16x2(d[r][1], 0.0f) & 0xFFFFu);
                }
            }
            cs[2 * c] = s0;
            cs[2 * c + 1] = s1;
        }
        if (c0 + kZGroup < kChunks) {
#pragma unroll
            for (int j = 0; j < 4 * kZGroup; ++j) zcur[j] = znext[j];
        }
    }
    if (BGRAD) {
        int lo = 0;  // first (chunk, column) index this lane still holds
#pragma unroll
        for (int st = 0; st < 3; ++st) {
            const int half = kChunks >> st;  // the lane holds 2 * half sums before the stage
            const bool upper = ((g8 >> st) & 1) != 0;
#pragma unroll
            for (int i = 0; i < half; ++i) {
                const float keep = upper ? cs[half + i] : cs[i];
                const float give = upper ? cs[i] : cs[half + i];
                cs[i] = keep + __shfl_xor_sync(0xffffffffu, give, 4 << st);
            }
            lo += upper ? half : 0;
        }
        // (chunk, column) indices lo .. lo + 3: chunks lo / 2 and lo / 2 + 1
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int v = lo + i;
            const int col = col0 + 8 * (v >> 1) + (v & 1);
            if (col < p.N) band[col] = cs[i];
        }
    }
}

// dgrad with the row cast of its output: dZ = acc * gelu'(Z) -> bf16 out as
// in store_dgrad, and the e5m2 codes and 1x128 scales of the stored bf16 dZ,
// blocked along N, exactly as the row cast would produce them from that
// output (the cast rule of cast_rule.cuh on the same bf16 values).  N % 128
// == 0, so the thread's half of the tile is one 128-column block of each of
// its four rows, and the block's 128 values sit with the four lanes of the
// thread's quad (32 each): the block amax is the quad's maximum.  A lane holds
// two codes of every 8-column chunk; two quad transposes give each lane the
// 32 contiguous codes of chunks 4 (lane % 4) .. +3 for two 16-byte stores.
template <bool ZSMEM>
__device__ __forceinline__ void store_dgrad_quant(const GemmParams& p, int row0, int col0,
                                                  const uint64_t (&acc)[4 * kChunks], int lane, const uint8_t* zrow) {
    uint16_t* out = static_cast<uint16_t*>(p.out);
    const uint16_t* zp = static_cast<const uint16_t*>(p.aux);
    const int g8 = lane >> 2;
    const int cq = lane & 3;
    uint32_t w[4 * kChunks];  // bf16 pairs of dZ, w[4c + r]
    float amax[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        uint32_t zw[4];
        if (ZSMEM)
            load_z_smem(zrow, g8, c, zw);
        else
            load_z_group(p, zp, true, row0, col0, c, zw);
        const int col = col0 + 8 * c;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float2 a = unpack_f32x2(acc[4 * c + r]);
            const float2 gd = dgelu_tanh2(bf16_lo(zw[r]), bf16_hi(zw[r]));
            const uint32_t v = pack_bf16x2(a.x * gd.x, a.y * gd.y);
            w[4 * c + r] = v;
            amax[r] = fmaxf(amax[r], fmaxf(fabsf(bf16_lo(v)), fabsf(bf16_hi(v))));
            const int row = row0 + 8 * r;
            if (row < p.M && col < p.N)
                *reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(row) * p.N + col) = v;
        }
    }
    const int cb = col0 - 2 * cq;  // first column of the thread's 128-column block
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        amax[r] = fmaxf(amax[r], __shfl_xor_sync(0xffffffffu, amax[r], 1));
        amax[r] = fmaxf(amax[r], __shfl_xor_sync(0xffffffffu, amax[r], 2));
        float inv, s;
        block_scale<1>(amax[r], inv, s);
        // codes of chunk 4g + e as 16-bit halves: lo = chunks 4g, 4g + 1; hi = 4g + 2, 4g + 3
        uint32_t lo[4], hi[4];
#pragma unroll
        for (int gq = 0; gq < 4; ++gq) {
            uint32_t h16[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t v = w[4 * (4 * gq + e) + r];
                h16[e] = encode2<1>(bf16_lo(v), bf16_hi(v), inv);
            }
            lo[gq] = h16[0] | (h16[1] << 16);
            hi[gq] = h16[2] | (h16[3] << 16);
        }
        // lane j receives group j's halves from every lane of the quad
        quad_transpose(lo, cq);
        quad_transpose(hi, cq);
        const int row = row0 + 8 * r;
        if (row < p.M && cb < p.N) {
            // chunk 4 cq + e: bytes of lanes 0..3 in order (each lane two codes)
            uint32_t o[8];
            o[0] = __byte_perm(lo[0], lo[1], 0x5410);
            o[1] = __byte_perm(lo[2], lo[3], 0x5410);
            o[2] = __byte_perm(lo[0], lo[1], 0x7632);
            o[3] = __byte_perm(lo[2], lo[3], 0x7632);
            o[4] = __byte_perm(hi[0], hi[1], 0x5410);
            o[5] = __byte_perm(hi[2], hi[3], 0x5410);
            o[6] = __byte_perm(hi[0], hi[1], 0x7632);
            o[7] = __byte_perm(hi[2], hi[3], 0x7632);
            uint4* dst = reinterpret_cast<uint4*>(p.qout + static_cast<int64_t>(row) * p.N + cb + 32 * cq);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
            if (cq == 0) p.qscale[static_cast<int64_t>(cb >> 7) * p.qsld + row] = s;
        }
    }
}

// -------------------------------------------------------------------- kernel

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_kernel(const __grid_constant__ TensorMaps maps, const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    SmemLayout& sm = *reinterpret_cast<SmemLayout*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                    ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t budget = p.budget_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_addr(&sm.full[s]), 1);
            mbar_init(smem_addr(&sm.empty[s]), 1);
        }
        for (int s = 0; s < kSStages; ++s) {
            mbar_init(smem_addr(&sm.sfull[s]), 1);
            mbar_init(smem_addr(&sm.sempty[s]), kEpiWarps);
        }
        for (int b = 0; b < kNumAcc; ++b) {
            mbar_init(smem_addr(&sm.acc_full[b]), 1);
            mbar_init(smem_addr(&sm.acc_empty[b]), kEpiWarps);
        }
        mbar_init(smem_addr(&sm.zfull), 1);
        mbar_init(smem_addr(&sm.zempty), kEpiWarps);
        mbar_init(smem_addr(&sm.drain), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&sm.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = sm.tmem_base;
    uint8_t* const zs = reinterpret_cast<uint8_t*>(&sm) + sizeof(SmemLayout);  // Z tile (dgrad only)
    const bool z_staged = uses_z<EPI>() && p.z_tma != 0;

    if (warp < kFirstEpiWarp) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtrl));
    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&maps.a);
            tma_prefetch_desc(&maps.b);
            tma_prefetch_desc(&maps.sa);
            tma_prefetch_desc(&maps.sb);
            int s = 0, ss = 0;
            uint32_t ph = 0, sph = 0;
            int n_issued = 0, ns_issued = 0;
            bool ok = true;
            if (!p.debug_starve) {
                for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
                    int g, mt, nt;
                    decode_tile(p, t, g, mt, nt);
                    const GroupEntry ge = p.groups[g];
                    const int m0 = mt * kBM, n0 = nt * kBN;
                    for (int kb = 0; kb < ge.nkb; ++kb) {
                        const int kbg = ge.kb_start + kb;
                        if (!mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1u, budget)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb = smem_addr(&sm.full[s]);
                        mbar_arrive_expect_tx(fb, kBM * kBK + kBN * kBK);
                        tma_load_2d(smem_addr(sm.a[s]), &maps.a, fb, kbg * kBK, m0);
                        tma_load_2d(smem_addr(sm.b[s]), &maps.b, fb, kbg * kBK, n0);
                        ++n_issued;
                        ring_advance<kStages>(s, ph);
                        if (!mbar_wait(smem_addr(&sm.sempty[ss]), sph ^ 1u, budget)) {
                            ok = false;
                            break;
                        }
                        const uint32_t sfb = smem_addr(&sm.sfull[ss]);
                        mbar_arrive_expect_tx(sfb, (kBM + kBN) * 4);
                        tma_load_2d(smem_addr(sm.sa[ss]), &maps.sa, sfb, m0, kbg);
                        tma_load_2d(smem_addr(sm.sb[ss]), &maps.sb, sfb, n0, kbg);
                        ++ns_issued;
                        ring_advance<kSStages>(ss, sph);
                    }
                }
            }
            if (ok) {
                // every stage must be released by its consumer before exit
                for (int i = 0; i < kStages; ++i) {
                    if (!mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1u, budget)) ok = false;
                    ring_advance<kStages>(s, ph);
                }
                for (int i = 0; i < kSStages; ++i) {
                    if (!mbar_wait(smem_addr(&sm.sempty[ss]), sph ^ 1u, budget)) ok = false;
                    ring_advance<kSStages>(ss, sph);
                }
            }
            if (!ok) {
                record_status(p.status, kStatusTimeout);
                // let the loads still in flight land before shared memory goes away
                for (int i = 1; i <= (n_issued < kStages ? n_issued : kStages); ++i) {
                    int si = s - i;
                    uint32_t pi = ph;
                    if (si < 0) {
                        si += kStages;
                        pi ^= 1u;
                    }
                    mbar_wait(smem_addr(&sm.full[si]), pi, budget);
                }
                for (int i = 1; i <= (ns_issued < kSStages ? ns_issued : kSStages); ++i) {
                    int si = ss - i;
                    uint32_t pi = sph;
                    if (si < 0) {
                        si += kSStages;
                        pi ^= 1u;
                    }
                    mbar_wait(smem_addr(&sm.sfull[si]), pi, budget);
                }
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------- Z tile loader (dgrad)
        if (z_staged && lane == 0) {
            tma_prefetch_desc(&maps.z);
            uint32_t zph = 0;
            int nz = 0;
            bool ok = true;
            if (!p.debug_starve) {
                for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
                    int g, mt, nt;
                    decode_tile(p, t, g, mt, nt);
                    // the previous tile's epilogue must have read the buffer
                    if (!mbar_wait(smem_addr(&sm.zempty), zph ^ 1u, budget)) {
                        ok = false;
                        break;
                    }
                    const uint32_t zb = smem_addr(&sm.zfull);
                    mbar_arrive_expect_tx(zb, kZBytes);
#pragma unroll
                    for (int j = 0; j < kBN / kZBoxCols; ++j)
                        tma_load_2d(smem_addr(zs + j * kZBoxBytes), &maps.z, zb, nt * kBN + j * kZBoxCols,
                                    mt * kBM);
                    ++nz;
                    zph ^= 1u;
                }
            }
            if (!ok) record_status(p.status, kStatusTimeout);
            // the last load must have landed before shared memory goes away
            if (nz > 0) mbar_wait(smem_addr(&sm.zfull), static_cast<uint32_t>(nz - 1) & 1u, budget);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        int s = 0, ab = 0;
        uint32_t ph = 0, aph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
            int g, mt, nt;
            decode_tile(p, t, g, mt, nt);
            const int nkb = p.groups[g].nkb;
            for (int kb = 0; kb < nkb; ++kb) {
                ok = mbar_wait_warp(smem_addr(&sm.acc_empty[ab]), aph ^ 1u, budget);
                if (ok) ok = mbar_wait_warp(smem_addr(&sm.full[s]), ph, budget);
                if (!ok) break;
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t d = tmem_base + static_cast<uint32_t>(ab * kBN);
                    const uint64_t adesc = smem_desc_k_sw128(smem_addr(sm.a[s]));
                    const uint64_t bdesc = smem_desc_k_sw128(smem_addr(sm.b[s]));
#pragma unroll
                    for (int k = 0; k < kBK / 32; ++k)
                        mma_f8f6f4(d, adesc + 2u * k, bdesc + 2u * k, p.idesc, k > 0 ? 1u : 0u);
                    mma_commit(smem_addr(&sm.empty[s]));
                    mma_commit(smem_addr(&sm.acc_full[ab]));
                }
                __syncwarp();
                ring_advance<kStages>(s, ph);
                ring_advance<kNumAcc>(ab, aph);
            }
        }
        if (!ok && lane == 0) record_status(p.status, kStatusTimeout);
        // all MMAs issued by this warp must complete before TMEM is released
        if (lane == 0) mma_commit(smem_addr(&sm.drain));
        __syncwarp();
        mbar_wait(smem_addr(&sm.drain), 0, budget);
        __syncwarp();
    } else if (warp >= kFirstEpiWarp) {
        // ------------------------------------------ promotion and epilogue
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
        const int ew = warp - kFirstEpiWarp;
        const int q = warp & 3;    // TMEM lane quadrant of this warp
        const int half = ew >> 2;  // which 128 columns of the tile
        const int g8 = lane >> 2;  // row within each 8-row group
        const int cq = lane & 3;   // column pair within each 8-column chunk
        int ab = 0, ss = 0;
        uint32_t aph = 0, sph = 0, zph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
            int g, mt, nt;
            decode_tile(p, t, g, mt, nt);
            const GroupEntry ge = p.groups[g];
            const int m0 = mt * kBM, n0 = nt * kBN;
            uint64_t acc[4 * kChunks];  // packed fp32 pairs, layout described above the stores
#pragma unroll
            for (int j = 0; j < 4 * kChunks; ++j) acc[j] = 0ull;
            const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                static_cast<uint32_t>(half * kHalfN);
            if (uses_z<EPI>() && !z_staged) {
                // the stored pre-activations of this tile are read once the K loop
                // is done: ask for them in L2 now (each lane of a quad one of the
                // quad's four rows; a row's 128 columns span at most three lines)
                const int prow = m0 + q * 32 + g8 + 8 * cq;
                const int pc0 = n0 + half * kHalfN;
                if (prow < p.M && pc0 < p.N) {
                    const uint16_t* zrow = static_cast<const uint16_t*>(p.aux) + static_cast<int64_t>(prow) * p.N;
                    const int pc1 = min(pc0 + kHalfN - 1, p.N - 1);
                    prefetch_l2(zrow + pc0);
                    prefetch_l2(zrow + min(pc0 + 64, pc1));
                    prefetch_l2(zrow + pc1);
                }
            }
            for (int kb = 0; kb < ge.nkb; ++kb) {
                ok = mbar_wait2_warp(smem_addr(&sm.acc_full[ab]), aph, smem_addr(&sm.sfull[ss]), sph, budget);
                if (!ok) break;
                tc_fence_after();
                const uint32_t tbuf = tq + static_cast<uint32_t>(ab * kBN);
                // row scales of the thread's four rows; column scales one pair per
                // chunk, shared by the four rows (one 8-byte load per 8 elements)
                uint64_t sa2[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float s = sm.sa[ss][q * 32 + g8 + 8 * r];
                    sa2[r] = pack_f32x2(s, s);
                }
                const float* sbp = &sm.sb[ss][half * kHalfN + 2 * cq];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint64_t plo[8], phi[8];
                    tmem_ld_16x256b_x4_pairs2(tbuf + 32u * h, tbuf + (16u << 16) + 32u * h, plo, phi);
                    if (h == 3) {
                        // the block's partial sums are all in registers: hand the buffer back
                        tc_fence_before();
                        __syncwarp();
                        mbar_arrive_lane0(smem_addr(&sm.acc_empty[ab]), lane);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int c = 4 * h + i;
                        const uint64_t sb = *reinterpret_cast<const uint64_t*>(sbp + 8 * c);
                        acc[4 * c + 0] = fma_f32x2(plo[2 * i], mul_f32x2(sa2[0], sb), acc[4 * c + 0]);
                        acc[4 * c + 1] = fma_f32x2(plo[2 * i + 1], mul_f32x2(sa2[1], sb), acc[4 * c + 1]);
                        acc[4 * c + 2] = fma_f32x2(phi[2 * i], mul_f32x2(sa2[2], sb), acc[4 * c + 2]);
                        acc[4 * c + 3] = fma_f32x2(phi[2 * i + 1], mul_f32x2(sa2[3], sb), acc[4 * c + 3]);
                    }
                }
                // the scale stage was read with ordinary loads and is refilled by
                // TMA: order the reads before the release (cross-proxy hazard)
                fence_proxy_async_smem();
                __syncwarp();
                mbar_arrive_lane0(smem_addr(&sm.sempty[ss]), lane);
                ring_advance<kNumAcc>(ab, aph);
                ring_advance<kSStages>(ss, sph);
            }
            if (!ok) break;
            const int row0 = m0 + q * 32 + g8;
            const int col0 = n0 + half * kHalfN + 2 * cq;
            if (EPI == kEpiWgrad) {
                store_wgrad(p, ge.out_index, row0, col0, acc);
            } else if (EPI == kEpiNone || EPI == kEpiBias || EPI == kEpiBiasGelu) {
                store_fprop<EPI>(p, row0, col0, acc);
            } else {
                // bias-gradient partials of this warp's 32 rows -> workspace band (4*mt + q)
                float* band = (EPI == kEpiDgeluBgrad) ? p.workspace + (static_cast<int64_t>(mt) * 4 + q) * p.N
                                                      : nullptr;
                if (z_staged) {
                    ok = mbar_wait_warp(smem_addr(&sm.zfull), zph, budget);
                    if (!ok) break;
                    const uint8_t* zrow = zs + half * (kHalfN / kZBoxCols) * kZBoxBytes + (q * 32 + g8) * 128 + 4 * cq;
                    if (EPI == kEpiDgeluQuant)
                        store_dgrad_quant<true>(p, row0, col0, acc, lane, zrow);
                    else
                        store_dgrad<EPI == kEpiDgeluBgrad, true>(p, row0, col0, acc, band, lane, zrow);
                    // read with ordinary loads, refilled by TMA: order before the release
                    fence_proxy_async_smem();
                    __syncwarp();
                    mbar_arrive_lane0(smem_addr(&sm.zempty), lane);
                    zph ^= 1u;
                } else if (EPI == kEpiDgeluQuant) {
                    store_dgrad_quant<false>(p, row0, col0, acc, lane, nullptr);
                } else {
                    store_dgrad<EPI == kEpiDgeluBgrad, false>(p, row0, col0, acc, band, lane, nullptr);
                }
            }
        }
        if (!ok && lane == 0) record_status(p.status, kStatusTimeout);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

template <int EPI>
int launch_gemm_impl(const TensorMaps& maps, const GemmParams& p, cudaStream_t stream, int grid) {
    auto kern = gemm_fp8_kernel<EPI>;
    static unsigned long long configured = 0;  // one bit per device ordinal
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -3;
    if (!(configured & (1ull << dev))) {
        // the register split above assumes exactly kLaunchRegs per thread at launch
        cudaFuncAttributes attr;
        if (cudaFuncGetAttributes(&attr, kern) != cudaSuccess || attr.numRegs != kLaunchRegs) return -3;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem_bytes<EPI>())) != cudaSuccess)
            return -3;
        configured |= 1ull << dev;
    }
    kern<<<grid, kThreads, smem_bytes<EPI>(), stream>>>(maps, p);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace fp8ll
